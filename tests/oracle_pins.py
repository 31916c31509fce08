"""Pins that tie the fp64 oracle to facts outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something fixed independently of its code: a library routine run on a
contiguous copy of the cache (torch's scaled-dot-product attention, scipy's
logsumexp), a closed form, or an invariant that any correct paged gather must
satisfy.  ``test_oracle_pins.py`` runs them against the real oracle and
against deliberately broken builds of it (every mutant must trip at least one
pin).

What the pins follow (the "mini-infer" pages):
  - prajwal7-2002 docs, "Systems Architecture" and "Core Capabilities at a
    Glance" (rows "Memory Allocation", "Batched Paged Decode", "Model
    Architecture"): physical 16-token block pool, per-request block table,
    direct physical gather with slot mapping, attention by SDPA.
  - psmarter write-up, feature list items 1 and 7: block-table
    PagedAttention, split-K flash decoding.
  - tom-jerr "Attention Backend" table: split-KV paged decode, page_size 256.
  - psmarter write-up, feature list items 3 and 5, and the prajwal7-2002
    docs' "Prompt Ingestion" row and speculative-decoding overview: several
    new tokens per sequence at once (chunked prefill, draft verification),
    read as causal attention over the pool.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from paged_kv_decode_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns through torch's own bf16 type (independent of the oracle's C)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def small_case(B=3, Hq=6, Hkv=2, D=32, bs=16, lens=(5, 16, 41), nb=24, seed=7, **kw):
    return W.make_workload("pin", B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=list(lens),
                           num_blocks=nb, seed=seed, write_new=False, **kw)


def contiguous_kv(w: W.DecodeWorkload, b: int):
    """Gather sequence b's K and V into contiguous [L, Hkv, D] fp64 arrays with numpy fancy indexing."""
    L = int(w.seq_lens[b])
    t = np.arange(L)
    phys = w.block_tables[b][t // w.block_size]
    off = t % w.block_size
    k = bf16_to_f64(w.k_cache)[phys, off]
    v = bf16_to_f64(w.v_cache)[phys, off]
    return k, v


def sdpa_reference(w: W.DecodeWorkload):
    """torch.nn.functional.scaled_dot_product_attention (fp64, CPU) on contiguous copies.

    The GQA group is expanded with repeat_interleave, i.e. query head h reads
    KV head h // (Hq / Hkv).
    """
    out = np.zeros((w.B, w.Hq, w.D))
    for b in range(w.B):
        L = int(w.seq_lens[b])
        if L == 0:
            continue
        k, v = contiguous_kv(w, b)
        q = torch.from_numpy(bf16_to_f64(w.q[b]))[:, None, :]            # [Hq, 1, D]
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(w.G, dim=0)  # [Hq, L, D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q, kt, vt, scale=float(w.scale))
        out[b] = o[:, 0, :].numpy()
    return out


def run_oracle(w: W.DecodeWorkload):
    return oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)


# ---------------------------------------------------------------- cache write
def pin_cache_write_index_put():
    """Scatter equals numpy index-put on a sentinel-filled pool; padding slots are skipped."""
    rng = np.random.default_rng(11)
    nb, bs, hkv, d = 8, 16, 2, 8
    sentinel = np.uint16(0xABCD)
    kc = np.full((nb, bs, hkv, d), sentinel, np.uint16)
    vc = np.full((nb, bs, hkv, d), sentinel, np.uint16)
    slots = np.array([5, -1, 127, 16, 64, -7, 3], np.int64)
    n = slots.shape[0]
    kn = rng.integers(0, 0xFFFF, (n, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 0xFFFF, (n, hkv, d), dtype=np.uint16)
    oracle.cache_write(kn, vn, slots, kc, vc)
    ek = np.full_like(kc, sentinel).reshape(nb * bs, hkv, d)
    ev = np.full_like(vc, sentinel).reshape(nb * bs, hkv, d)
    ok = slots >= 0
    ek[slots[ok]] = kn[ok]
    ev[slots[ok]] = vn[ok]
    assert np.array_equal(kc.reshape(nb * bs, hkv, d), ek), "K scatter differs from index-put"
    assert np.array_equal(vc.reshape(nb * bs, hkv, d), ev), "V scatter differs from index-put"


def pin_cache_write_then_gather():
    """After the write, the gather through the block table returns the new token at L-1."""
    w = W.make_workload("pin", B=3, Hq=4, Hkv=2, D=16, block_size=16, seq_lens=[1, 16, 35],
                        num_blocks=12, seed=5)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.cache_write(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    for b in range(w.B):
        t = int(w.seq_lens[b]) - 1
        p = w.block_tables[b, t // w.block_size]
        assert np.array_equal(kc[p, t % w.block_size], w.k_new[b])
        assert np.array_equal(vc[p, t % w.block_size], w.v_new[b])


def pin_cache_write_rejects_bad_slots():
    kc = np.zeros((2, 16, 1, 8), np.uint16)
    vc = kc.copy()
    kn = np.ones((2, 1, 8), np.uint16)
    for bad in ([3, 3], [0, 32]):
        try:
            oracle.cache_write(kn, kn, np.array(bad, np.int64), kc, vc)
        except oracle.OracleError:
            continue
        raise AssertionError(f"slots {bad} accepted")


# ------------------------------------------------------------ gather + SDPA
def pin_sdpa_contiguous():
    """Oracle equals torch SDPA on a contiguous gathered cache (several shapes) to 1e-12."""
    cases = [
        small_case(),
        small_case(B=2, Hq=8, Hkv=8, D=16, lens=(33, 7), nb=8, seed=3),           # MHA, G=1
        small_case(B=2, Hq=7, Hkv=1, D=64, lens=(64, 1), nb=6, seed=4),           # G=7
        small_case(B=2, Hq=4, Hkv=2, D=16, bs=256, lens=(300, 513), nb=6, seed=9),  # 256-token pages
        small_case(B=1, Hq=12, Hkv=4, D=24, bs=32, lens=(95,), nb=5, seed=12),
    ]
    for w in cases:
        out, _ = run_oracle(w)
        ref = sdpa_reference(w)
        err = np.abs(out - ref).max()
        assert err < 1e-12, f"{w.Hq}/{w.Hkv}/{w.D}/bs{w.block_size}: oracle vs SDPA {err}"


def pin_permutation_invariance():
    """Relabelling physical blocks (pool permuted, tables remapped) leaves the output bit-identical."""
    w = small_case(B=3, Hq=6, Hkv=3, D=16, lens=(20, 48, 3), nb=10, seed=21)
    out, lse = run_oracle(w)
    perm = np.random.default_rng(1).permutation(w.num_blocks)   # new position of old block i
    inv = np.argsort(perm)
    k2 = w.k_cache[inv]
    v2 = w.v_cache[inv]
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.decode(w.q, k2, v2, bt2, w.seq_lens, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


# --------------------------------------------------------------- closed forms
def pin_single_token_returns_v():
    """L = 1: the softmax weight is 1, out is the V row exactly and lse is the single score."""
    w = small_case(B=2, Hq=4, Hkv=2, D=32, lens=(1, 1), nb=4, seed=31)
    out, lse = run_oracle(w)
    for b in range(w.B):
        p = w.block_tables[b, 0]
        for h in range(w.Hq):
            g = h // w.G
            v = bf16_to_f64(w.v_cache[p, 0, g])
            assert np.array_equal(out[b, h], v), "L=1 output is not the V row"
            s = float(w.scale) * float(bf16_to_f64(w.q[b, h]) @ bf16_to_f64(w.k_cache[p, 0, g]))
            assert abs(lse[b, h] - s) < 1e-12


def pin_identical_keys_mean():
    """All keys equal: uniform weights, out = mean of the V rows, lse = s + ln L."""
    w = small_case(B=2, Hq=4, Hkv=2, D=16, lens=(23, 40), nb=8, seed=41)
    w.k_cache[:] = w.k_cache[0, 0][None, None]
    out, lse = run_oracle(w)
    for b in range(w.B):
        k, v = contiguous_kv(w, b)
        L = int(w.seq_lens[b])
        for h in range(w.Hq):
            g = h // w.G
            assert np.abs(out[b, h] - v[:, g].mean(axis=0)).max() < 1e-12
            s = float(w.scale) * float(bf16_to_f64(w.q[b, h]) @ k[0, g])
            assert abs(lse[b, h] - (s + math.log(L))) < 1e-12


def pin_scale_zero_mean():
    """scale = 0: every score is 0, out = mean of V regardless of K, lse = ln L."""
    w = small_case(B=2, Hq=6, Hkv=3, D=8, lens=(9, 33), nb=8, seed=51, scale=0.0)
    out, lse = run_oracle(w)
    for b in range(w.B):
        _, v = contiguous_kv(w, b)
        for h in range(w.Hq):
            assert np.abs(out[b, h] - v[:, h // w.G].mean(axis=0)).max() < 1e-12
            assert abs(lse[b, h] - math.log(int(w.seq_lens[b]))) < 1e-12


def pin_two_token_closed_form():
    """Golden fixture: two keys with scores 0 and 1 give weights 1/(1+e), e/(1+e)."""
    with open(os.path.join(GOLDEN, "two_token.json")) as f:
        fx = json.load(f)
    D = len(fx["q"])
    kc = np.zeros((1, 16, 1, D), np.uint16)
    vc = np.zeros((1, 16, 1, D), np.uint16)
    kc[0, 0, 0] = f64_to_bf16_bits(fx["k0"])
    kc[0, 1, 0] = f64_to_bf16_bits(fx["k1"])
    vc[0, 0, 0] = f64_to_bf16_bits(fx["v0"])
    vc[0, 1, 0] = f64_to_bf16_bits(fx["v1"])
    q = f64_to_bf16_bits(fx["q"]).reshape(1, 1, D)
    out, lse = oracle.decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([2], np.int32),
                             fx["scale"])
    e = math.e
    expect = (np.array(fx["v0"]) + e * np.array(fx["v1"])) / (1 + e)
    assert np.abs(out[0, 0] - expect).max() < 1e-14
    assert abs(lse[0, 0] - math.log(1 + e)) < 1e-14


def pin_linearity_pow2():
    """Scaling V by 2 scales the output by 2 exactly (a power of two commutes with rounding)."""
    w = small_case(seed=61)
    out, lse = run_oracle(w)
    vb = bf16_to_f64(w.v_cache) * 2.0
    v2 = f64_to_bf16_bits(vb)
    out2, lse2 = oracle.decode(w.q, w.k_cache, v2, w.block_tables, w.seq_lens, w.scale)
    assert np.array_equal(out2, 2.0 * out) and np.array_equal(lse, lse2)


def pin_identical_q_heads():
    """Query heads of one group with the same q give bit-identical outputs; different groups differ."""
    w = small_case(B=2, Hq=8, Hkv=2, D=16, lens=(30, 17), nb=8, seed=71)
    w.q[:] = w.q[:, :1]
    out, _ = run_oracle(w)
    for b in range(w.B):
        for g in range(w.Hkv):
            grp = out[b, g * w.G:(g + 1) * w.G]
            assert np.array_equal(grp, np.broadcast_to(grp[0], grp.shape))
        assert not np.array_equal(out[b, 0], out[b, w.G]), "KV heads not distinguished"


def pin_lse_logsumexp():
    """lse equals scipy.special.logsumexp of the scores computed by numpy einsum."""
    from scipy.special import logsumexp
    w = small_case(B=2, Hq=4, Hkv=2, D=32, lens=(50, 3), nb=6, seed=81)
    _, lse = run_oracle(w)
    for b in range(w.B):
        k, _ = contiguous_kv(w, b)
        q = bf16_to_f64(w.q[b])
        kk = np.repeat(k, w.G, axis=1)                      # [L, Hq, D]
        s = float(w.scale) * np.einsum("hd,lhd->hl", q, kk)
        assert np.abs(lse[b] - logsumexp(s, axis=1)).max() < 1e-12


def pin_empty_sequence():
    """L = 0 reads nothing: out = 0 and lse = -inf."""
    w = small_case(B=2, Hq=2, Hkv=1, D=8, lens=(0, 4), nb=3, seed=91)
    out, lse = run_oracle(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


def pin_poison_never_read():
    """NaN in every pool row attention must not read leaves the output unchanged."""
    w = small_case(B=3, Hq=4, Hkv=2, D=16, lens=(5, 17, 32), nb=9, seed=101)
    clean, _ = run_oracle(w)
    wp = small_case(B=3, Hq=4, Hkv=2, D=16, lens=(5, 17, 32), nb=9, seed=101, poison_unused=True)
    out, _ = run_oracle(wp)
    assert np.array_equal(out, clean)


# ------------------------------------------------------------------- split-KV
def pin_split_combine_equals_unsplit():
    """Partials over any block-aligned (or not) partition, merged by LSE, equal unsplit to 1e-12."""
    w = small_case(B=3, Hq=6, Hkv=2, D=16, lens=(1, 70, 129), nb=20, seed=111)
    out, lse = run_oracle(w)
    for P, chunk in ((1, 160), (2, 80), (3, 48), (9, 16), (19, 7), (40, 16)):
        po, pl = oracle.decode_partial(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                       w.scale, P, chunk)
        o2, l2 = oracle.combine(po, pl)
        assert np.abs(o2 - out).max() < 1e-12, f"P={P} chunk={chunk}"
        assert np.abs(l2 - lse).max() < 1e-12


def pin_combine_closed_form():
    """Two partials with lse 0 and ln 3 weigh 1/4 and 3/4; an empty (-inf) partial weighs 0."""
    po = np.array([[[1.0, -2.0], [5.0, 6.0], [123.0, 456.0]]])
    pl = np.array([[0.0, math.log(3.0), -math.inf]])
    out, lse = oracle.combine(po, pl)
    assert np.abs(out[0] - np.array([0.25 * 1 + 0.75 * 5, 0.25 * -2 + 0.75 * 6])).max() < 1e-15
    assert abs(lse[0] - math.log(4.0)) < 1e-15
    out, lse = oracle.combine(np.zeros((1, 2, 3)), np.full((1, 2), -math.inf))
    assert np.all(out == 0) and np.isneginf(lse[0])


def pin_partial_ranges():
    """A partial covering tokens [a, b) equals SDPA over exactly those tokens."""
    w = small_case(B=1, Hq=2, Hkv=1, D=16, lens=(45,), nb=4, seed=121)
    po, pl = oracle.decode_partial(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                   w.scale, 3, 16)
    k, v = contiguous_kv(w, 0)
    for p, (a, bnd) in enumerate(((0, 16), (16, 32), (32, 45))):
        q = torch.from_numpy(bf16_to_f64(w.q[0]))[:, None, :]
        kt = torch.from_numpy(k[a:bnd]).permute(1, 0, 2)
        vt = torch.from_numpy(v[a:bnd]).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(q, kt, vt, scale=float(w.scale))
        assert np.abs(po[0, :, p] - o[:, 0].numpy()).max() < 1e-12


# ------------------------------------------------------ multi-query (causal)
def causal_scores_and_sdpa(w: W.DecodeWorkload):
    """torch SDPA (fp64, CPU) with an explicit boolean causal mask on contiguous
    copies, plus numpy scores for the log-sum-exp.  Query i of sequence b sits at
    position L - q_len + i and sees tokens [0, L - q_len + i]; a query at a
    negative position sees nothing (expected output 0, lse -inf)."""
    from scipy.special import logsumexp
    out = np.zeros((w.B, w.q_len, w.Hq, w.D))
    lse = np.full((w.B, w.q_len, w.Hq), -np.inf)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        if L == 0:
            continue
        k, v = contiguous_kv(w, b)                                         # [L, Hkv, D]
        qf = bf16_to_f64(w.q[b])                                           # [q_len, Hq, D]
        q = torch.from_numpy(qf).permute(1, 0, 2)                           # [Hq, q_len, D]
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        pos = L - w.q_len + np.arange(w.q_len)
        mask = np.arange(L)[None, :] <= pos[:, None]                       # [q_len, L]
        seen = mask.any(axis=1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, kt, vt, attn_mask=torch.from_numpy(mask), scale=float(w.scale))
        o = o.permute(1, 0, 2).numpy()                                     # [q_len, Hq, D]
        out[b][seen] = o[seen]
        kg = np.repeat(k, w.G, axis=1)                                     # [L, Hq, D]
        s = np.einsum("ihd,thd->iht", qf, kg) * w.scale                    # [q_len, Hq, L]
        for i in np.nonzero(seen)[0]:
            lse[b, i] = logsumexp(s[i][:, mask[i]], axis=1)
    return out, lse


def run_oracle_mq(w: W.DecodeWorkload):
    return oracle.decode_mq(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)


def pin_mq_sdpa_causal():
    """Multi-query oracle equals masked SDPA (output) and logsumexp (lse) to 1e-12."""
    cases = [
        small_case(q_len=3),
        small_case(B=2, Hq=4, Hkv=4, D=16, lens=(33, 5), nb=6, seed=31, q_len=4),         # G=1
        small_case(B=3, Hq=7, Hkv=1, D=32, lens=(20, 1, 2), nb=6, seed=32, q_len=3),      # L < q_len
        small_case(B=2, Hq=4, Hkv=2, D=16, bs=256, lens=(300, 7), nb=4, seed=33, q_len=5),
        small_case(B=1, Hq=6, Hkv=2, D=24, lens=(70,), nb=6, seed=34, q_len=16),
    ]
    for w in cases:
        out, lse = run_oracle_mq(w)
        ref, ref_lse = causal_scores_and_sdpa(w)
        err = np.abs(out - ref).max()
        assert err < 1e-12, f"q_len {w.q_len} G {w.G}: oracle vs masked SDPA {err}"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse)), "lse -inf pattern differs"
        assert np.abs(lse[fin] - ref_lse[fin]).max() < 1e-12, "lse differs from logsumexp"


def pin_mq_negative_positions_see_nothing():
    """Queries at positions < 0 (L < q_len) give a zero row and lse = -inf."""
    w = small_case(B=2, Hq=2, Hkv=1, D=8, lens=(2, 0), nb=3, seed=35, q_len=4)
    out, lse = run_oracle_mq(w)
    assert np.all(out[0, :2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(np.isfinite(lse[0, 2:]))
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    # position 0 sees exactly token 0: its V row, bit for bit after widening
    k, v = contiguous_kv(w, 0)
    assert np.array_equal(out[0, 2], np.repeat(v[0], w.G, axis=0))   # head h reads KV head h // G


def pin_mq_last_query_is_decode():
    """The last query (position L - 1) sees the whole sequence: it equals the
    single-query decode of the same rows, and q_len = 1 is decode itself."""
    w = small_case(B=3, Hq=6, Hkv=2, D=16, lens=(9, 33, 16), nb=8, seed=36, q_len=3)
    out, lse = run_oracle_mq(w)
    out1, lse1 = oracle.decode(np.ascontiguousarray(w.q[:, -1]), w.k_cache, w.v_cache,
                               w.block_tables, w.seq_lens, w.scale)
    assert np.array_equal(out[:, -1], out1) and np.array_equal(lse[:, -1], lse1)
    # query i equals the decode of the sequence truncated to L - q_len + i + 1 tokens
    for i in range(w.q_len):
        lens_i = (w.seq_lens - w.q_len + i + 1).astype(np.int32)
        oi, li = oracle.decode(np.ascontiguousarray(w.q[:, i]), w.k_cache, w.v_cache,
                               w.block_tables, lens_i, w.scale)
        assert np.array_equal(out[:, i], oi) and np.array_equal(lse[:, i], li)


# ------------------------------------------------------------------ FP8 KV
# ("Mini-Infer: A High-Performance LLM Inference Acceleration Engine for
# Production Environments", section "Memory Optimization and KV Cache
# Management": several quantisation schemes; read as OCP e4m3 with one fp32
# scale per pool.)  torch's float8_e4m3fn is the independent reference.
def _torch_e4m3(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)


def pin_fp8_widen_every_code():
    """All 256 codes widen to bf16 exactly as torch's e4m3 type does (NaN codes to NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_bf16(codes)
    ref = _torch_e4m3(codes).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(_torch_e4m3(codes).float().numpy())
    assert list(codes[nan]) == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(bf16_to_f64(got[nan])))


def pin_fp8_quantise_matches_torch_in_range():
    """bf16 / scale (fp32) rounded to e4m3 equals torch's cast, bit for bit, inside +-448,
    including values exactly halfway between codes (ties to even) and subnormals."""
    rng = np.random.default_rng(41)
    vals = [rng.standard_normal(4000) * 3, rng.standard_normal(1000) * 1e-2,
            rng.uniform(-440, 440, 1000)]
    w = _torch_e4m3(np.arange(0x7F, dtype=np.uint8)).float().numpy().astype(np.float64)
    mids = (w[1:] + w[:-1]) / 2                                     # halfway points (exact in bf16)
    x = np.concatenate(vals + [mids, -mids])
    bits = f64_to_bf16_bits(x)
    for scale in (1.0, 0.0625, 0.37):
        got = oracle.bf16_to_e4m3(bits, scale)
        xf = torch.from_numpy(bf16_to_f64(bits)).float() / torch.tensor(scale, dtype=torch.float32)
        inside = xf.abs() <= 448
        ref = xf.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got[inside.numpy()], ref[inside.numpy()]), f"scale {scale}"


def pin_fp8_quantise_saturates_and_round_trips():
    """Beyond +-448 the code saturates to +-448; NaN stays NaN; every finite code
    survives widen-then-quantise with scale 1."""
    big = f64_to_bf16_bits(np.array([449.0, 1e4, -3e5, -449.0]))
    assert list(oracle.bf16_to_e4m3(big, 1.0)) == [0x7E, 0x7E, 0xFE, 0xFE]
    nan = np.array([0x7FC0], np.uint16)
    assert oracle.bf16_to_e4m3(nan, 1.0)[0] & 0x7F == 0x7F
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(oracle.bf16_to_e4m3(oracle.e4m3_to_bf16(codes), 1.0), codes)


def pin_fp8_decode_equals_sdpa_on_dequantised_cache():
    """Attention over e4m3 pools equals SDPA over torch-dequantised contiguous K/V
    (code * scale in fp64, with the fp32 pool scales the library receives, the
    softmax scale applied as given): the factored scales agree to fp64 rounding."""
    w = small_case(B=3, Hq=6, Hkv=2, D=32, lens=(5, 16, 41), nb=24, seed=51)
    ks, vs = 0.043, 0.029
    k8 = oracle.bf16_to_e4m3(w.k_cache, ks)
    v8 = oracle.bf16_to_e4m3(w.v_cache, vs)
    out, lse = oracle.decode_fp8(w.q, k8, v8, w.block_tables, w.seq_lens, w.scale, ks, vs)
    kd = _torch_e4m3(k8).double().numpy() * float(np.float32(ks))
    vd = _torch_e4m3(v8).double().numpy() * float(np.float32(vs))
    for b in range(w.B):
        L = int(w.seq_lens[b])
        t = np.arange(L)
        phys, off = w.block_tables[b][t // w.block_size], t % w.block_size
        kt = torch.from_numpy(kd[phys, off]).permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        vt = torch.from_numpy(vd[phys, off]).permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        q = torch.from_numpy(bf16_to_f64(w.q[b]))[:, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(q, kt, vt, scale=float(w.scale))
        err = np.abs(out[b] - o[:, 0].numpy()).max()
        assert err < 1e-12, f"fp8 decode vs dequantised SDPA: {err}"


def pin_fp8_cache_write_quantises_the_new_rows():
    """The fp8 write stores exactly bf16_to_e4m3 of each new row at its slot."""
    w = W.make_workload("pin", B=3, Hq=4, Hkv=2, D=16, block_size=16, seq_lens=[1, 16, 35],
                        num_blocks=12, seed=52)
    kc = np.full(w.k_cache.shape, 0x11, np.uint8)
    vc = np.full(w.v_cache.shape, 0x22, np.uint8)
    oracle.cache_write_fp8(w.k_new, w.v_new, w.slot_mapping, kc, vc, 0.5, 0.25)
    ek = np.full_like(kc, 0x11).reshape(-1, w.Hkv, w.D)
    ev = np.full_like(vc, 0x22).reshape(-1, w.Hkv, w.D)
    ek[w.slot_mapping] = _torch_e4m3_from(w.k_new, 0.5)
    ev[w.slot_mapping] = _torch_e4m3_from(w.v_new, 0.25)
    assert np.array_equal(kc.reshape(ek.shape), ek) and np.array_equal(vc.reshape(ev.shape), ev)


def _torch_e4m3_from(bits: np.ndarray, scale: float) -> np.ndarray:
    x = torch.from_numpy(bf16_to_f64(bits)).float() / torch.tensor(scale, dtype=torch.float32)
    return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
