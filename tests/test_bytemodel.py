"""The algorithmic byte model against the payload arithmetic the pages print."""
import os

from verify_attention_gb300 import bytemodel as bm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture():
    out = {}
    for line in open(os.path.join(GOLDEN, "kv_payload_bytes.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            out[k] = int(v)
    return out


def test_payload_per_token_layer():
    f = _fixture()
    assert bm.kv_bytes_per_token_layer(8, 128, 1) // 1 == f["kv_values_per_token_layer"]
    assert bm.kv_bytes_per_token_layer(8, 128, 2) == f["bf16_bytes_per_token_layer"]
    assert bm.kv_bytes_per_token_layer(8, 128, 1) == f["fp8_bytes_per_token_layer"]


def test_payload_aggregates():
    f = _fixture()
    for layers, key in ((48, "48_layers"), (54, "54_layers")):
        assert layers * bm.kv_bytes_per_token_layer(8, 128, 2) / 1024 == f[f"bf16_kib_per_token_{key}"]
        assert layers * bm.kv_bytes_per_token_layer(8, 128, 1) / 1024 == f[f"fp8_kib_per_token_{key}"]
    # TP4 KV-head sharding: 2 of the 8 heads per rank, 54 layers
    assert 54 * bm.kv_bytes_per_token_layer(2, 128, 2) / 1024 == f["bf16_kib_per_token_per_rank_tp4"]
    assert 54 * bm.kv_bytes_per_token_layer(2, 128, 1) / 1024 == f["fp8_kib_per_token_per_rank_tp4"]


def test_attention_bytes_sliding_window_span():
    # window 512 (window_left 511) with 12 verifier rows sees 523 distinct keys
    assert bm.visible_keys_any_row(4096, 12, 511) == 523
    assert bm.visible_keys_any_row(300, 12, 511) == 300
    b = bm.attention_bytes([4096], 12, 72, 8, 128, 1, -1, 64)
    assert b == 4096 * 2048 + 2 * 12 * 72 * 128 * 2 + 4 * 65 + 4 + 8
    # per-row visibility sums to the flop count
    assert bm.attention_flops([10], 3, 1, 1, 1) == 4 * (2 + 2 + 2)
