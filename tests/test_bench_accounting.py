"""The algorithmic bytes the bench divides by, for the attention and decoder workloads,
against the shapes they come from (CPU; no GPU)."""
import bench


def test_attention_step_bytes():
    # int4 weights with one fp16 scale per 32: 4.5 bits per weight
    assert bench.WQKV_BYTES == (32 + 2 * 4) * 128 * 2048 * 9 // 16 == 5_898_240
    assert bench.WO_BYTES == 2048 * 32 * 128 * 9 // 16 == 4_718_592
    row = 4 * 128 * 2  # one position of every key/value head, bf16
    fixed = bench.WQKV_BYTES + bench.WO_BYTES + 2 * row + 3 * 2048 * 2
    assert bench.attn_step_bytes(32768, 0) == fixed + 32768 * 2 * row
    # a window attends min(window, positions) keys
    assert bench.attn_step_bytes(32768, 513) == fixed + 513 * 2 * row
    assert bench.attn_step_bytes(100, 513) == fixed + 100 * 2 * row
    assert bench.attn_name(32768, 0) == "attn_decode_ctx32768_full"
    assert bench.attn_name(32768, 513) == "attn_decode_ctx32768_swa513"


def test_decoder_layer_kinds():
    kinds = bench.decoder_kinds(49)
    full = [l for l, (w, rope) in enumerate(kinds) if w == 0]
    assert len(full) == 14 and len(kinds) - len(full) == 35
    assert all(not rope for w, rope in kinds if w == 0)
    assert all(rope and w == 513 for w, rope in kinds if w != 0)
