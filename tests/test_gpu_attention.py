"""GPU parity of the causal prefill attention (apr_prefill_attention) against
the float64 oracle (aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs:
qwen35_prefill_attention / qwen35_attention_pass for what is computed,
qwen35_flash_prefill_attention for the fp16-input fused form).

Tolerance, from the arithmetic of the fused form (q, k and v rounded to fp16,
the softmax weights rounded to fp16 for the value product, fp32 accumulation):
* against the exact attention of the f32 inputs: relative Frobenius <= 2e-3,
  the bar of the fp16-input projections;
* against the oracle on fp16-rounded q, k, v: every element within
  2^-9 * max|v| over the visible values. A weight rounded to fp16 is off by at
  most 2^-11 of itself, which moves a weighted mean of values by at most
  2 * 2^-11 * max|v|; the fp32 sums add far less.
Bit for bit where the definition makes the result exact: the first position
(one visible key, weight exactly 1) gives fp16(v_0), also when the call cuts
the query tiles' key ranges into parts; splitting a chunk into two calls
changes no row when neither call cuts key ranges (with parts, a row's sums
are grouped by the call's shape: equal within the bars above, not bit for
bit).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_guards, dev, errors, guarded

pytestmark = pytest.mark.gpu

D = 256
REL = 2e-3
F16_IN_OVER_VMAX = 2.0 ** -9


def run(q, c, Q=None, T=None, pos0=None):
    Q = c["Q"] if Q is None else Q
    T = c["T"] if T is None else T
    pos0 = c["pos0"] if pos0 is None else pos0
    nh = c["num_heads"]
    buf, out = guarded(T, nh * D)
    q.apr_prefill_attention(dev(Q), dev(c["K"]), dev(c["V"]), out, T, pos0, nh, c["num_kv_heads"], D)
    q.apr_stream_status()
    check_guards(buf, T, nh * D)
    return out.cpu().numpy()


def assert_attention(y, c, rows=None):
    args = (c["Q"], c["K"], c["V"], c["T"], c["pos0"], c["num_heads"], c["num_kv_heads"], D)
    ref = oracle.prefill_attention_f64(*args, rows=rows)
    r16 = oracle.prefill_attention_f16_inputs_f64(*args, rows=rows)
    rel, _, _ = errors(y, ref)
    assert rel <= REL, f"rel-Frobenius {rel:.3e} > {REL}"
    last = c["pos0"] + (c["T"] if rows is None else int(np.max(rows)) + 1)
    vmax = float(np.abs(c["V"][:last].astype(np.float16).astype(np.float64)).max())
    mx = float(np.abs(np.asarray(y, np.float64) - r16).max())
    assert mx <= F16_IN_OVER_VMAX * vmax, f"max|err| vs fp16 inputs {mx:.3e} > 2^-9 * {vmax:.3f}"
    return rel, mx / vmax


# (T, pos0, num_heads, num_kv_heads): one row, ragged query tiles, a chunk
# ending exactly on a 64-key tile, key tiles past the first query tile, a long
# cache before the chunk, MHA, MQA and the 9B model's 16 / 4 grouping
SHAPES = [(1, 0, 2, 1), (5, 0, 2, 1), (128, 0, 1, 1), (129, 0, 4, 2), (200, 37, 4, 2), (300, 130, 2, 2),
          (3, 61, 16, 4), (1, 64, 2, 2), (64, 900, 2, 1), (130, 4000, 2, 1)]


@pytest.mark.parametrize("T,pos0,nh,nkv", SHAPES)
def test_attention_matches_oracle(q, T, pos0, nh, nkv):
    c = synth.attention_case(T, pos0, nh, nkv, seed=T + pos0)
    assert_attention(run(q, c), c)


@pytest.mark.parametrize("T,nh,nkv", [(4, 4, 2), (1024, 2, 1)])
def test_first_position_takes_its_own_value_exactly(q, T, nh, nkv):
    # 1024 rows over 2 heads: 16 CTAs, the longest over 16 key tiles, so the
    # key tiles are cut into parts of one and row 0 goes through the
    # combination (its other part sees no key)
    c = synth.attention_case(T, 0, nh, nkv, seed=21)
    y = run(q, c)
    v16 = c["V"].astype(np.float16).astype(np.float32)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.array_equal(y[0, h * D:(h + 1) * D], v16[0, g * D:(g + 1) * D]), h


def test_zero_query_averages_the_visible_values(q):
    c = synth.attention_case(70, 10, 2, 1, seed=22)
    c["Q"] = np.zeros_like(c["Q"])
    y = run(q, c).astype(np.float64)
    v16 = c["V"].astype(np.float16).astype(np.float64)
    mean = np.cumsum(v16, axis=0) / np.arange(1, len(v16) + 1)[:, None]
    for t in range(70):
        for h in range(2):
            # uniform weights 1 over the visible keys: only the fp32 sums round
            # (a key too many or too few would move the mean by about 1 / count)
            np.testing.assert_allclose(y[t, h * D:(h + 1) * D], mean[10 + t, :D], rtol=0,
                                       atol=1e-4 * np.abs(v16).max())


def test_cache_rows_past_the_chunk_are_never_read(q):
    # 70 rows of NaN after position pos0 + T - 1: any read of them would show
    c = synth.attention_case(150, 20, 2, 1, seed=23)
    y = run(q, c)
    c2 = dict(c)
    for key in ("K", "V"):
        c2[key] = np.concatenate([c[key], np.full((70, c[key].shape[1]), np.nan, np.float32)])
    assert np.array_equal(run(q, c2), y)


@pytest.mark.parametrize("pos0", [200, 1000])
def test_rescale_of_the_running_sum(q, pos0):
    # one key per 64-key tile whose score grows by 6 (8.7 in base 2) from tile
    # to tile: the reference max moves at every tile (at pos0 = 1000 the key
    # tiles are cut into parts whose maxima differ by as much)
    T, nh, nkv = 256, 2, 1
    c = synth.attention_case(T, pos0, nh, nkv, seed=24)
    u = np.zeros(D, np.float32)
    u[0] = 1.0
    c["Q"][:, :] = np.tile(16.0 * u, nh)[None, :]
    for i in range((pos0 + T) // 64):
        c["K"][64 * i + 5, :] = np.tile(6.0 * i * u, nkv)
    assert_attention(run(q, c), c)


def test_splitting_a_chunk_changes_no_row(q):
    # rows 0..99 at pos0, then rows 100..299 at pos0 + 100, over the same
    # cache; 64 query heads, so that no call cuts its key ranges into parts
    c = synth.attention_case(300, 40, 64, 4, seed=25)
    whole = run(q, c)
    a = run(q, c, Q=c["Q"][:100], T=100)
    b = run(q, c, Q=c["Q"][100:], T=200, pos0=140)
    assert np.array_equal(np.concatenate([a, b]), whole)


def test_repeat_is_bitwise_identical(q):
    c = synth.attention_case(257, 33, 4, 4, seed=26)
    assert np.array_equal(run(q, c), run(q, c))


def test_empty_chunk_writes_nothing(q):
    out = torch.full((4, 2 * D), 7.0, device="cuda")
    z = torch.zeros(16, device="cuda")
    q.apr_prefill_attention(z, z, z, out, 0, 5, 2, 1, D)
    q.apr_stream_status()
    assert bool((out == 7.0).all())


def test_key_parts_of_a_late_chunk(q):
    # the last 256 rows of a 2048-token prompt (pos0 = 1792): 32 CTAs of up to
    # 32 key tiles become parts of a few tiles each, then combined
    c = synth.attention_case(256, 1792, 16, 4, seed=28)
    y = run(q, c)
    rows = np.array([0, 1, 63, 64, 127, 128, 200, 255])
    assert_attention(y[rows], c, rows=rows)
    assert np.array_equal(run(q, c), y)


@pytest.mark.parametrize("T", [512, 2048])
def test_nine_b_chunk_sampled_rows(q, T):
    # the 9B model's attention (16 query heads over 4 KV heads, head_dim 256)
    # at its chunk sizes; rows sampled across the query tiles, every head
    c = synth.attention_case(T, 0, 16, 4, seed=27)
    y = run(q, c)
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, T - 1], rng.choice(T, 40, replace=False)]))
    assert_attention(y[rows], c, rows=rows)
