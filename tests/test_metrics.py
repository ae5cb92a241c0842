"""The bench's byte counting against the numbers the KBench
megakernel_int4_weight_decode.py spec prints for a batch-1 decode step of its
3B int4-g128 model: 1,920,133,120 bytes per step (codes + scales/zeros + KV
cache) and a 197 MB packed LM head."""
from weight_only_bit_w4a16_gb300 import metrics, synth


def test_decode_step_bytes_match_the_spec():
    d, ffn, hd = synth.DECODER["d"], synth.DECODER["ffn"], synth.DECODER["hd"]
    n_q, n_kv, vocab = synth.DECODER["n_q"], synth.DECODER["n_kv"], synth.DECODER["vocab"]
    layers, prefix, steps = 28, 2048, 32
    per_layer = [(n_q * hd, d), (n_kv * hd, d), (n_kv * hd, d), (d, n_q * hd),
                 (ffn, d), (ffn, d), (d, ffn)]
    w = layers * sum(metrics.weight_bytes("int4", N, K, 128) for N, K in per_layer)
    w += metrics.weight_bytes("int4", vocab, d, 128)            # tied LM head
    # KV cache read by attention: (prefix + decode steps) tokens, k and v, bf16
    kv = (prefix + steps) * layers * 2 * n_kv * hd * 2
    assert w + kv == 1_920_133_120


def test_lm_head_packed_bytes():
    N, K = synth.LAYER_SHAPES["lm_head"]
    assert N * K // 2 == 197_001_216


def test_call_bytes_and_flops():
    # decode GEMV: A, codes, bf16 scales, zeros, C
    assert metrics.call_bytes("int4", 1, 8192, 3072, 128) == \
        2 * 3072 + 8192 * 1536 + 8192 * 24 * 2 + 8192 * 24 + 8192 * 2
    assert metrics.call_bytes("nvfp4", 16, 256, 512, 16, "fp32") == \
        2 * 16 * 512 + 256 * 256 + 256 * 32 + 16 * 256 * 4
    assert metrics.call_flops(2048, 3072, 3072) == 2 * 2048 * 3072 * 3072
