"""The benchmark's roofline numerators on the CPU: the algorithmic bytes and
flops bench.py divides by the measured times, against closed forms from the
70B config (every weight read once, KV once per KV head, new K/V written once;
2 flops per multiply-add, attention 4 d flops per visible (query, key, q-head)
pair)."""

import bench
from llama_decoder_layer_gb300 import inputs as I


def _params(spec):
    d, H, I_ = spec.head_dim, spec.hidden, spec.intermediate
    return ((spec.n_heads + 2 * spec.n_kv_heads) * d * H + H * spec.n_heads * d + 2 * I_ * H + H * I_ + 2 * H)


def test_70b_layer_weight_bytes():
    spec = I.SPECS["decode_70b"]
    bl = I.make_batch(spec, 0, "cpu")
    alg = bench.layer_algorithmic(spec, bl)
    # 80 q/kv heads x 128 x 8192 + 8192 x 8192 + 3 x 28672 x 8192 + two norm weights, bf16
    assert _params(spec) == 855_654_400
    assert alg["weight_bytes"] == 2 * 855_654_400  # 1.71 GB per layer


def test_70b_decode_kv_and_total_bytes():
    spec = I.SPECS["decode_70b"]
    bl = I.make_batch(spec, 0, "cpu")
    alg = bench.layer_algorithmic(spec, bl)
    nkv, d = spec.n_kv_heads, spec.head_dim
    kv_read = sum(c + q for c, q in zip(bl.ctx_lens, bl.q_lens)) * nkv * d * 2 * 2
    kv_write = bl.num_tokens * nkv * d * 2 * 2
    assert alg["kv_bytes"] == kv_read + kv_write
    assert alg["bytes"] == alg["weight_bytes"] + alg["kv_bytes"] + alg["act_bytes"]
    assert 3.5e9 < alg["bytes"] < 4.5e9  # the ~3.9 GB the decode line divides by


def test_70b_prefill_flops():
    spec = I.SPECS["prefill_70b"]
    bl = I.make_batch(spec, 0, "cpu")
    alg = bench.layer_algorithmic(spec, bl)
    T = bl.num_tokens
    pairs = 8 * sum(range(1, 4097))  # causal (query, key) pairs of 8 fresh 4096-token sequences
    assert alg["flops"] == 2 * T * _params(spec) + 4 * spec.head_dim * pairs * spec.n_heads
    assert abs(alg["flops"] / 1e12 - 58.3) < 0.1  # the 58.3 TFLOP of the prefill line


def test_gate_up_launch_flops():
    spec = I.SPECS["stack_70b"]
    T = I.make_batch(spec, 0, "cpu").num_tokens
    assert T == 4128
    assert abs(2.0 * T * 2 * spec.intermediate * spec.hidden - 3.878e12) < 1e9  # flops_per_launch
