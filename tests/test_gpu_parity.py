"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (Dev, assert_close, assert_lse_close, bf16_dev_to_f64, oracle_after_write,
                      u16_to_dev_bf16)
from paged_kv_decode_cache_gb300 import pa
from paged_kv_decode_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_decode_cache_gb300 import build
    build.build()


def kernels_for(Hq, Hkv, D):
    """The decode kernels that can run this shape (both are tested where both can)."""
    G = Hq // Hkv
    ks = []
    if G <= 8:
        ks.append("cuda_core")
    if D == 128 and G <= 32:
        ks.append("tensor_core")
    return ks


# ---------------------------------------------------------------- cache write
def test_cache_write_bit_exact_with_sentinels():
    rng = np.random.default_rng(0)
    nb, bs, hkv, d = 40, 16, 8, 128
    sentinel = np.uint16(0x5A5A)
    kc = np.full((nb, bs, hkv, d), sentinel, np.uint16)
    vc = np.full((nb, bs, hkv, d), sentinel, np.uint16)
    slots = rng.choice(nb * bs, 300, replace=False).astype(np.int64)
    slots[::7] = -1                               # padding
    kn = rng.integers(0, 0xFFFF, (300, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 0xFFFF, (300, hkv, d), dtype=np.uint16)
    dk, dv = u16_to_dev_bf16(kc), u16_to_dev_bf16(vc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write(u16_to_dev_bf16(kn), u16_to_dev_bf16(vn), torch.from_numpy(slots).cuda(),
                      dk, dv, status=status)
    oracle.cache_write(kn, vn, slots, kc, vc)
    gk = dk.view(torch.int16).cpu().numpy().view(np.uint16)
    gv = dv.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    assert status.item() == 0


def test_cache_write_out_of_pool_slot_is_skipped_and_reported():
    nb, bs, hkv, d = 4, 16, 2, 64
    kc = np.zeros((nb, bs, hkv, d), np.uint16)
    slots = np.array([3, nb * bs + 5, 10], np.int64)
    kn = np.full((3, hkv, d), 0x3F80, np.uint16)
    dk, dv = u16_to_dev_bf16(kc), u16_to_dev_bf16(kc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write(u16_to_dev_bf16(kn), u16_to_dev_bf16(kn), torch.from_numpy(slots).cuda(),
                      dk, dv, status=status)
    assert status.item() & pa.PA_STATUS_BAD_SLOT
    ref = kc.copy()
    oracle.cache_write(kn[[0, 2]], kn[[0, 2]], slots[[0, 2]], ref, ref.copy())
    assert np.array_equal(dk.view(torch.int16).cpu().numpy().view(np.uint16), ref)


# ------------------------------------------------------- decode, small shapes
SMALL = [
    # (Hq, Hkv, D, bs, lens)
    (4, 2, 64, 16, (1, 17, 33, 100)),
    (8, 8, 128, 16, (1, 15, 16, 17, 31, 33)),       # G = 1
    (12, 2, 128, 16, (48, 130, 7)),                 # G = 6
    (28, 4, 128, 16, (257, 16, 1)),                 # G = 7
    (16, 2, 128, 16, (64, 65)),                     # G = 8
    (6, 2, 64, 16, (200, 3)),                       # G = 3
    (10, 2, 128, 32, (95, 64, 1)),                  # G = 5, 32-token blocks
    (16, 4, 128, 256, (300, 513, 256, 1)),          # 256-token pages
    (4, 1, 64, 256, (1000,)),                       # G = 4, pages, long-ish
    (2, 2, 128, 16, (0, 5)),                        # empty sequence
    (32, 2, 128, 16, (129, 300)),                   # G = 16 (tensor cores only)
    (48, 2, 128, 16, (200, 65)),                    # G = 24: one KV head per CTA, 32 columns
    (24, 2, 128, 256, (700, 1)),                    # G = 12, pages (tensor cores only)
    (8, 2, 128, 16, (127, 128, 129, 255, 256, 257)),  # chunk boundaries of 128 tokens
]


def _small(Hq, Hkv, D, bs, lens, seed=0, **kw):
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    return W.make_workload("small", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                           seq_lens=list(lens), num_blocks=nb, seed=seed, **kw)


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-D{c[2]}-bs{c[3]}")
def test_decode_small_elementwise(case, use_kernel):
    w = _small(*case, seed=hash(case) % 1000, poison_unused=True)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    for kernel in kernels_for(w.Hq, w.Hkv, w.D):
        use_kernel(kernel)
        dev = Dev(w)
        dev.write()
        out, lse = dev.decode()
        assert_close(bf16_dev_to_f64(out), ref, f"pa_decode {kernel}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"pa_decode {kernel}")
        for P in (2, 3, 7):
            so, sl, _ = dev.splitkv(P)
            assert_close(bf16_dev_to_f64(so), ref, f"splitkv P={P} {kernel}")
            assert_lse_close(sl.cpu().double().numpy(), ref_lse, f"splitkv P={P} {kernel}")
        assert dev.status_value() == 0


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("P", [1, 2, 5, 16, 40])
def test_partials_match_oracle_partials(P, kernel, use_kernel):
    use_kernel(kernel)
    w = _small(12, 2, 128, 16, (1, 70, 129, 400), seed=P)
    dev = Dev(w)
    dev.write()
    kc, vc = oracle_after_write(w)
    chunk = pa.pa_partition_tokens(w.max_blocks, w.block_size, P)
    po, pl = dev.partial(P)
    ro, rl = oracle.decode_partial(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, P, chunk)
    assert_close(po.cpu().double().numpy(), ro, "partial o")
    assert_lse_close(pl.cpu().double().numpy(), rl, "partial lse")


@pytest.mark.parametrize("lens,P", [((1500,), 33), ((1500,), 100), ((1500,), 150), ((700, 1500), 60),
                                    ((2100,), 64), ((2100,), 65), ((2100,), 128)])
def test_fused_merge_many_partitions(lens, P, use_kernel):
    """More than 32 partitions per row (the merge's partition-parallel tasks),
    some of them empty past the sequence end; few sequences, so the cooperative
    grid fits and the merge runs inside the decode launch."""
    w = _small(12, 2, 128, 16, lens, seed=P)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    for kernel in kernels_for(w.Hq, w.Hkv, w.D):
        use_kernel(kernel)
        dev = Dev(w)
        dev.write()
        so, sl, _ = dev.splitkv(P)
        assert_close(bf16_dev_to_f64(so), ref, f"splitkv P={P} {kernel}")
        assert_lse_close(sl.cpu().double().numpy(), ref_lse, f"splitkv P={P} {kernel}")
        assert dev.status_value() == 0


@pytest.mark.parametrize("P", [2, 3, 4, 5])
def test_split_grid_in_waves(P, use_kernel):
    """A split grid that runs in waves (200 sequences of all 8 KV heads per CTA:
    200 CTAs per partition on 152 SMs): partials, then the combine kernel.
    Lengths from 0 to 300 leave some partitions empty; a second call on the
    same workspace gives the same result, and the fused step and FP8 pools
    take the same path."""
    use_kernel("auto")
    rng = np.random.default_rng(70 + P)
    lens = [int(x) for x in rng.integers(0, 301, size=200)]
    w = _small(16, 8, 128, 16, lens, seed=P, poison_unused=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pa.pa_decode_launches(w.B, 1, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size, P, sms) == 2
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)), dtype=torch.uint8,
                     device="cuda")
    for rep in range(2):
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_splitkv(out, lse, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws, status=dev.status)
        assert_close(bf16_dev_to_f64(out), ref, f"P={P} call {rep}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"P={P} call {rep}")
    assert dev.status_value() == 0
    # the fused write + decode
    dev2 = Dev(w)
    so, sl, _ = dev2.step(P)
    assert_close(bf16_dev_to_f64(so), ref, f"step P={P}")
    assert_lse_close(sl.cpu().double().numpy(), ref_lse, f"step P={P}")
    assert dev2.status_value() == 0
    # FP8 pools
    w8 = W.with_fp8_pools(w)
    ref8, ref8_lse = oracle.decode_fp8(w8.q, w8.k_cache8, w8.v_cache8, w8.block_tables, w8.seq_lens,
                                       w8.scale, w8.k_scale, w8.v_scale)
    kc8, vc8 = _fp8_dev(w8)
    ws.zero_()
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitkv_fp8(out, lse, dev.q, kc8, vc8, w8.k_scale, w8.v_scale, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws, status=dev.status)
    assert_close(bf16_dev_to_f64(out), ref8, f"fp8 P={P}")
    assert_lse_close(lse.cpu().double().numpy(), ref8_lse, f"fp8 P={P}")
    assert dev.status_value() == 0


@pytest.mark.parametrize("Hkv", [1, 2])
@pytest.mark.parametrize("P", [257, 300])
def test_more_partitions_than_the_in_launch_merge_holds(P, Hkv, use_kernel):
    """More than 256 partitions of one sequence (CUDA-core kernel, D = 64, whose
    small CTAs let such a grid be resident at once): the in-launch merge holds
    at most 256 partitions per row, so these partials are merged by the
    combine kernel instead; no partition may be dropped."""
    use_kernel("cuda_core")
    L = 16 * P - 5                       # 16-token partitions, the last one ragged
    w = _small(2 * Hkv, Hkv, 64, 16, (L,), seed=P + Hkv)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    assert pa.pa_partition_tokens(w.max_blocks, w.block_size, P) == 16
    so, sl, _ = dev.splitkv(P)
    assert_close(bf16_dev_to_f64(so), ref, f"splitkv P={P}")
    assert_lse_close(sl.cpu().double().numpy(), ref_lse, f"splitkv P={P}")
    assert dev.status_value() == 0


def test_combine_matches_oracle():
    g = torch.Generator().manual_seed(3)
    B, Hq, P, D = 3, 5, 9, 128
    po = torch.randn(B, Hq, P, D, generator=g, dtype=torch.float64).float()
    pl = (torch.randn(B, Hq, P, generator=g, dtype=torch.float64) * 4).float()
    pl[0, 0, :] = -math.inf                       # all partitions empty
    pl[1, 2, 3:] = -math.inf                      # some empty
    po[pl == -math.inf] = 0
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    pa.pa_combine(out, lse, po.cuda(), pl.cuda())
    ro, rl = oracle.combine(po.double().numpy(), pl.double().numpy())
    assert_close(bf16_dev_to_f64(out), ro, "combine")
    assert_lse_close(lse.cpu().double().numpy(), rl, "combine")


# ----------------------------------------------------- workloads at full size
FULL = ["tiny", "qwen2.5-1.5b-B1", "qwen2.5-1.5b-B8", "qwen2.5-7b-bs16", "qwen2.5-7b-bs256",
        "long-B1-L4096", "long-B2-L4096", "long-B1-L32768", "long-B2-L32768", "qwen3-0.6b-B256"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size(name, use_kernel):
    """The bench's launch configuration (the fused step: auto kernel, auto split),
    then split and unsplit decode with each kernel forced, on the full-size
    workload, every (b, h) row against the oracle."""
    w = W.WORKLOADS[name]()
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    fused = Dev(w)
    out_f, lse_f, Pf = fused.step(0)
    assert fused.status_value() == 0
    gk, gv = fused.pools()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc), f"{name}: pools after the step"
    assert_close(bf16_dev_to_f64(out_f), ref, f"{name} step P={Pf}")
    assert_lse_close(lse_f.cpu().double().numpy(), ref_lse, f"{name} step P={Pf}")
    del fused
    dev = Dev(w)
    dev.write()
    for kernel in ["auto"] + kernels_for(w.Hq, w.Hkv, w.D):
        use_kernel(kernel)
        out_s, lse_s, P = dev.splitkv(0)
        out_u, lse_u = dev.decode()
        assert dev.status_value() == 0
        for tag, o, l in (("splitkv", out_s, lse_s), ("decode", out_u, lse_u)):
            assert_close(bf16_dev_to_f64(o), ref, f"{name} {tag} {kernel} P={P}")
            assert_lse_close(l.cpu().double().numpy(), ref_lse, f"{name} {tag} {kernel}")


# ------------------------------------------------------ bit-exact invariants
@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_block_permutation_invariance_bit_exact(kernel, use_kernel):
    use_kernel(kernel)
    w = _small(28, 4, 128, 16, (300, 77, 16), seed=5)
    dev = Dev(w)
    out1, lse1 = dev.decode()
    perm = np.random.default_rng(2).permutation(w.num_blocks)
    inv = np.argsort(perm)
    w2 = _small(28, 4, 128, 16, (300, 77, 16), seed=5)
    w2.k_cache = w.k_cache[inv].copy()
    w2.v_cache = w.v_cache[inv].copy()
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)],
                               -1).astype(np.int32)
    out2, lse2 = Dev(w2).decode()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_single_token_returns_v_row_exactly(kernel, use_kernel):
    use_kernel(kernel)
    w = _small(8, 2, 128, 16, (1, 1, 1), seed=9)
    dev = Dev(w)
    dev.write()
    out, _ = dev.decode()
    o2, _, _ = dev.splitkv(3)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.B):
        for h in range(w.Hq):
            assert np.array_equal(got[b, h], w.v_new[b, h // w.G])
    assert torch.equal(out, o2)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_value_scaling_by_two_is_exact(kernel, use_kernel):
    use_kernel(kernel)
    w = _small(12, 2, 128, 16, (100, 33), seed=11)
    out1, lse1 = Dev(w).decode()
    v2 = torch.from_numpy(w.v_cache.view(np.int16)).view(torch.bfloat16).float() * 2
    w.v_cache = v2.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out2, lse2 = Dev(w).decode()
    assert torch.equal(out2.float(), out1.float() * 2) and torch.equal(lse1, lse2)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_identical_query_heads_give_identical_outputs(kernel, use_kernel):
    use_kernel(kernel)
    w = _small(16, 2, 128, 16, (90, 40), seed=13)
    w.q[:] = w.q[:, :1]
    out, _ = Dev(w).decode()
    for g in range(w.Hkv):
        grp = out[:, g * w.G:(g + 1) * w.G]
        assert torch.equal(grp, grp[:, :1].expand_as(grp))


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_poisoned_pool_rows_never_leak(kernel, use_kernel):
    use_kernel(kernel)
    lens = (5, 17, 250)
    clean = Dev(_small(12, 2, 128, 16, lens, seed=17)).decode()[0]
    poisoned = Dev(_small(12, 2, 128, 16, lens, seed=17, poison_unused=True)).decode()[0]
    assert torch.isfinite(poisoned.float()).all()
    assert torch.equal(clean, poisoned)


# ---------------------------------------------------------- bad device data
@pytest.mark.parametrize("shape", [(4, 2, 64), (14, 2, 128)])
def test_bad_block_id_is_reported_not_dereferenced(shape):
    w = _small(*shape, 16, (40, 20), seed=19)
    w.block_tables[0, 1] = w.num_blocks + 1000
    w.block_tables[1, 0] = -5
    dev = Dev(w)
    out, _ = dev.decode()
    torch.cuda.synchronize()
    assert dev.status_value() & pa.PA_STATUS_BAD_BLOCK


@pytest.mark.parametrize("shape", [(4, 2, 64), (14, 2, 128)])
def test_bad_seq_len_is_reported_and_clamped(shape):
    w = _small(*shape, 16, (40, 20), seed=23)
    w.seq_lens = np.array([40, 10_000], np.int32)
    dev = Dev(w)
    dev.decode()
    torch.cuda.synchronize()
    assert dev.status_value() & pa.PA_STATUS_BAD_SEQLEN


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_fused_merge_reuses_its_workspace(kernel, use_kernel):
    """Consecutive split calls on one workspace give the same result, and the merge
    counters at the end of the workspace are back at zero after every call."""
    use_kernel(kernel)
    w = _small(28, 4, 128, 16, (700, 300, 33), seed=31)
    dev = Dev(w)
    P = 5
    nbytes = pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws)
        torch.cuda.synchronize()
        counters = ws[-(((w.B * w.Hq * 8 + 255) // 256) * 256):]
        assert int(counters.count_nonzero()) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref, _ = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    assert_close(bf16_dev_to_f64(outs[0]), ref, f"fused merge {kernel}")


# ----------------------------------------------------- fused write + decode
STEP_CASES = [
    (28, 4, 128, 16, (4096, 700, 33, 1)),
    (12, 2, 128, 16, (1, 17, 512, 2000)),
    (16, 8, 128, 16, (129, 2048, 1000)),
    (16, 4, 128, 256, (300, 513, 256, 1)),
    (4, 2, 64, 16, (1, 17, 33, 100)),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-D{c[2]}-bs{c[3]}")
@pytest.mark.parametrize("P", [1, 3, 0])
def test_decode_step_equals_write_then_decode(case, P, use_kernel):
    """pa_decode_step gives bit-for-bit the result of pa_cache_write followed by
    pa_decode_splitkv, leaves the pools exactly as the oracle's cache write does,
    and matches the oracle within tolerance."""
    w = _small(*case, seed=sum(case[4]) % 997, poison_unused=True)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    for kernel in kernels_for(w.Hq, w.Hkv, w.D):
        use_kernel(kernel)
        fused = Dev(w)
        out_f, lse_f, Pf = fused.step(P)
        two = Dev(w)
        two.write()
        out_t, lse_t, _ = two.splitkv(Pf)
        torch.cuda.synchronize()
        assert fused.status_value() == 0 and two.status_value() == 0
        assert torch.equal(out_f, out_t) and torch.equal(lse_f, lse_t), f"{kernel} P={Pf}"
        gk, gv = fused.pools()
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc), f"{kernel}: pools differ"
        assert_close(bf16_dev_to_f64(out_f), ref, f"pa_decode_step {kernel} P={Pf}")
        assert_lse_close(lse_f.cpu().double().numpy(), ref_lse, f"pa_decode_step {kernel}")


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_decode_step_refuses_a_slot_it_does_not_read(kernel, use_kernel):
    """A slot that is not position L - 1 of its sequence is not written and is reported;
    a negative slot is skipped silently."""
    use_kernel(kernel)
    w = _small(8, 2, 128, 16, (40, 20, 70), seed=37)
    w.slot_mapping[0] = (w.slot_mapping[0] + 3) % (w.num_blocks * w.block_size)  # wrong position
    w.slot_mapping[1] = -1                                                    # padding
    dev = Dev(w)
    k0, v0 = dev.pools()
    dev.step(2)
    torch.cuda.synchronize()
    assert dev.status_value() & pa.PA_STATUS_BAD_SLOT
    gk, gv = dev.pools()
    kc, vc = k0.copy(), v0.copy()
    oracle.cache_write(w.k_new[2:], w.v_new[2:], w.slot_mapping[2:], kc, vc)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


def test_splitkv_small_workspace_is_rejected():
    w = _small(12, 2, 128, 16, (300,), seed=29)
    dev = Dev(w)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=4, workspace=ws)
    assert e.value.code == pa.PA_EWORKSPACE


# ------------------------------------------------------------ graph capture
def test_decode_step_replays_in_a_cuda_graph():
    w = W.qwen25_1p5b(8)
    dev = Dev(w)
    P = pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
    ws = torch.zeros(pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dev.write()
        pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    eager = out.clone()
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.pa_cache_write(dev.k_new, dev.v_new, dev.slot_mapping, dev.k_cache, dev.v_cache)
        pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


# ------------------------------------------- multi-query (causal) decode
MQ_SMALL = [
    # (Hq, Hkv, D, bs, lens, q_len)
    (8, 8, 128, 16, (1, 15, 16, 17, 40), 4),        # G = 1, all 4 queries in one CTA
    (12, 2, 128, 16, (48, 130, 7), 2),              # G = 6
    (28, 4, 128, 16, (257, 16, 3), 4),              # G = 7: 2 query groups
    (16, 8, 128, 16, (200, 129, 5), 8),             # G = 2, 16 columns per head
    (32, 2, 128, 16, (129, 300), 3),                # G = 16: one query per CTA
    (16, 4, 128, 256, (300, 513, 2), 5),            # pages; L < q_len
    (6, 2, 128, 16, (70, 33), 16),                  # G = 3: 5 queries per CTA, 4 groups
]


@pytest.mark.parametrize("case", MQ_SMALL, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-bs{c[3]}-q{c[5]}")
def test_mq_small_elementwise(case):
    Hq, Hkv, D, bs, lens, q_len = case
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    w = W.make_workload("mq", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=list(lens),
                        num_blocks=nb, seed=sum(lens) + q_len, poison_unused=True, q_len=q_len)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (1, 2, 3, 7, 0):
        out, lse, Pu = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"pa_decode_mq P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"pa_decode_mq P={Pu}")
    assert dev.status_value() == 0


# More query columns per KV head than the decode kernel holds (q_len * G > 32):
# the prefill-shaped kernel, 128 query rows per CTA.
MQ_PREFILL = [
    # (Hq, Hkv, bs, lens, q_len)
    (8, 8, 16, (1, 40, 200), 64),        # G = 1: 128 positions per tile; L < q_len
    (28, 4, 16, (300, 64, 129), 40),     # G = 7: 18 positions (126 rows) per tile, 3 tiles
    (64, 2, 16, (500, 37), 9),           # G = 32: 4 positions per tile
    (12, 2, 256, (700, 513), 100),       # G = 6, 256-token pages
    (6, 2, 16, (1000,), 200),            # G = 3: 42 positions per tile, 5 tiles
    (16, 8, 16, (17, 15), 33),           # G = 2, every sequence shorter than q_len
    (16, 2, 16, (129, 191, 64), 65),     # G = 8: chunk and tile boundaries
]


@pytest.mark.parametrize("case", MQ_PREFILL, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-bs{c[2]}-q{c[4]}")
def test_mq_prefill_shape_elementwise(case):
    Hq, Hkv, bs, lens, q_len = case
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    w = W.make_workload("pf", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, block_size=bs, seq_lens=list(lens),
                        num_blocks=nb, seed=sum(lens) + q_len, poison_unused=True, q_len=q_len)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (1, 2, 3, 7, 0):
        out, lse, Pu = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"prefill-shaped mq P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"prefill-shaped mq P={Pu}")
    assert dev.status_value() == 0


def test_mq_prefill_shape_reports_a_bad_block():
    """A bad block id inside a prefill-shaped call is reported and never read."""
    w = W.make_workload("pfbad", B=2, Hq=28, Hkv=4, D=128, block_size=16, seq_lens=[300, 200],
                        num_blocks=40, seed=9, q_len=40)
    w.block_tables[0, 3] = w.num_blocks + 7
    w.block_tables[1, 1] = -3
    dev = Dev(w)
    out, lse, _ = dev.mq(1)
    torch.cuda.synchronize()
    assert dev.status_value() & pa.PA_STATUS_BAD_BLOCK
    assert torch.isfinite(out.float()).all()


def test_mq_single_query_is_splitkv_bit_exact():
    w = W.make_workload("mq1", B=3, Hq=28, Hkv=4, D=128, block_size=16, seq_lens=[300, 17, 1024],
                        num_blocks=100, seed=5, q_len=1)
    dev = Dev(w)
    dev.write()
    for P in (1, 4):
        o1, l1, _ = dev.splitkv(P)
        q = dev.q.view(w.B, 1, w.Hq, w.D)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)),
                         dtype=torch.uint8, device="cuda")
        o2 = torch.empty((w.B, 1, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        l2 = torch.empty((w.B, 1, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_mq(o2, l2, q, dev.k_cache, dev.v_cache, dev.block_tables, dev.seq_lens,
                        w.scale, num_splits=P, workspace=ws)
        assert torch.equal(o1, o2[:, 0]) and torch.equal(l1, l2[:, 0]), f"P={P}"


def test_mq_chunk_of_64_queries():
    """A small prefill-like chunk: 64 new tokens per sequence, G = 7 (32 query groups)."""
    w = W.make_workload("chunk", B=2, Hq=28, Hkv=4, D=128, block_size=16, seq_lens=[600, 64],
                        num_blocks=48, seed=77, q_len=64)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (1, 3):
        out, lse, _ = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"chunk P={P}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"chunk P={P}")


@pytest.mark.parametrize("B", [1, 8])
def test_mq_chunk_of_512_queries_qwen25_1p5b(B):
    """A 512-token chunked-prefill chunk per sequence on the Qwen2.5-1.5B-shaped
    layer (Hq = 12, Hkv = 2, the context including the chunk ~ U[512, 2048]):
    auto split and unsplit, every row against the oracle."""
    lens = W._uniform_lens(2002 + B, B, 512, 2048)
    nb = sum((L + 15) // 16 for L in lens) + 8
    w = W.make_workload("chunk512", B=B, Hq=12, Hkv=2, D=128, block_size=16, seq_lens=lens,
                        num_blocks=nb, max_blocks=128, seed=512 + B, q_len=512)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (0, 1):
        out, lse, Pu = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"chunk512 B={B} P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"chunk512 B={B} P={Pu}")
    assert dev.status_value() == 0


@pytest.mark.parametrize("name", ["qwen2.5-1.5b-B8-spec4", "qwen2.5-7b-bs16-spec4",
                                  "qwen3-0.6b-B256-spec4"])
def test_mq_workload_full_size(name):
    """The bench's launch configuration (auto P) and unsplit, against the oracle."""
    w = W.WORKLOADS[name]()
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (0, 1):
        out, lse, Pu = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"{name} P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"{name} P={Pu}")
    assert dev.status_value() == 0


# ------------------------------------------------------------- FP8 (e4m3) pools
def _fp8_dev(w):
    """Device copies of an FP8 workload's pools (uint8 codes)."""
    return (torch.from_numpy(w.k_cache8).cuda(), torch.from_numpy(w.v_cache8).cuda())


def test_fp8_cache_write_bit_exact():
    """The quantising write equals the oracle's, byte for byte, on sentinel pools:
    ordinary values, ties, tiny values, values past +-448 * scale and infinities."""
    rng = np.random.default_rng(8)
    nb, bs, hkv, d = 30, 16, 4, 128
    n = 200
    slots = rng.choice(nb * bs, n, replace=False).astype(np.int64)
    slots[::9] = -1
    x = rng.standard_normal((2, n, hkv, d)) * 3
    x[:, ::5] *= 1e-3                                   # subnormal codes
    x[:, 1::7] *= 400                                   # saturation
    bits = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bits[0, 3, 0, :4] = [0x7F80, 0xFF80, 0x0000, 0x8000]  # +inf, -inf, +0, -0
    kn, vn = bits[0].copy(), bits[1].copy()
    ks, vs = 0.0625, 0.011
    kc = np.full((nb, bs, hkv, d), 0x5A, np.uint8)
    vc = np.full((nb, bs, hkv, d), 0xA5, np.uint8)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write_fp8(u16_to_dev_bf16(kn), u16_to_dev_bf16(vn), torch.from_numpy(slots).cuda(),
                          dk, dv, ks, vs, status=status)
    oracle.cache_write_fp8(kn, vn, slots, kc, vc, ks, vs)
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    assert status.item() == 0


FP8_SMALL = [
    # (Hq, Hkv, bs, lens)
    (8, 8, 16, (1, 15, 16, 17, 33)),                # G = 1
    (28, 4, 16, (257, 16, 1)),                      # G = 7
    (16, 8, 16, (200, 129, 5)),                     # G = 2
    (32, 2, 16, (129, 300)),                        # G = 16
    (16, 4, 256, (300, 513, 2)),                    # pages
    (2, 2, 16, (0, 5)),                             # empty sequence
    (64, 4, 16, (100, 257, 31)),                    # G = 16, 4 heads per CTA (MMA N = 64)
    (32, 1, 16, (140, 64)),                         # G = 32, one head per CTA (MMA N = 64)
]


@pytest.mark.parametrize("case", FP8_SMALL, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-bs{c[2]}")
def test_fp8_decode_small_elementwise(case):
    Hq, Hkv, bs, lens = case
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    w = W.with_fp8_pools(W.make_workload("f8", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, block_size=bs,
                                         seq_lens=list(lens), num_blocks=nb, seed=sum(lens) + 3,
                                         poison_unused=True, write_new=False))
    ref, ref_lse = oracle.decode_fp8(w.q, w.k_cache8, w.v_cache8, w.block_tables, w.seq_lens,
                                     w.scale, w.k_scale, w.v_scale)
    dev = Dev(w)
    kc, vc = _fp8_dev(w)
    for P in (1, 2, 3, 7, 0):
        Pu = P or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, Pu)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_splitkv_fp8(out, lse, dev.q, kc, vc, w.k_scale, w.v_scale, dev.block_tables,
                                 dev.seq_lens, w.scale, num_splits=Pu, workspace=ws,
                                 status=dev.status)
        assert_close(bf16_dev_to_f64(out), ref, f"fp8 P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"fp8 P={Pu}")
    assert dev.status_value() == 0


@pytest.mark.parametrize("P", [33, 64, 100, 140])
def test_fp8_merge_many_partitions(P):
    """FP8 pools with more than 32 partitions per row: the sixteen-warp CTAs
    share each merge task between ceil(P / 32) warps and several tasks at once."""
    lens = (2390,)  # one sequence: every partition's CTA is resident at once
    w = W.with_fp8_pools(W.make_workload("f8m", B=1, Hq=28, Hkv=4, D=128, block_size=16,
                                         seq_lens=list(lens), num_blocks=160, seed=P,
                                         write_new=False))
    ref, ref_lse = oracle.decode_fp8(w.q, w.k_cache8, w.v_cache8, w.block_tables, w.seq_lens,
                                     w.scale, w.k_scale, w.v_scale)
    dev = Dev(w)
    kc, vc = _fp8_dev(w)
    ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitkv_fp8(out, lse, dev.q, kc, vc, w.k_scale, w.v_scale, dev.block_tables,
                             dev.seq_lens, w.scale, num_splits=P, workspace=ws, status=dev.status)
    assert_close(bf16_dev_to_f64(out), ref, f"fp8 P={P}")
    assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"fp8 P={P}")
    assert dev.status_value() == 0


@pytest.mark.parametrize("name", ["qwen2.5-7b-bs16-fp8", "qwen3-0.6b-B256-fp8", "long-B2-L32768-fp8"])
def test_fp8_workload_full_size(name):
    """Write this step's tokens with pa_cache_write_fp8, then decode (auto P and
    unsplit), against the oracle's write and decode."""
    w = W.WORKLOADS[name]()
    kc8, vc8 = w.k_cache8.copy(), w.v_cache8.copy()
    oracle.cache_write_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, w.k_scale, w.v_scale)
    ref, ref_lse = oracle.decode_fp8(w.q, kc8, vc8, w.block_tables, w.seq_lens, w.scale,
                                     w.k_scale, w.v_scale)
    dev = Dev(w)
    kc, vc = _fp8_dev(w)
    pa.pa_cache_write_fp8(dev.k_new, dev.v_new, dev.slot_mapping, kc, vc, w.k_scale, w.v_scale,
                          status=dev.status)
    assert np.array_equal(kc.cpu().numpy(), kc8) and np.array_equal(vc.cpu().numpy(), vc8)
    for P in (0, 1):
        Pu = P or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, Pu)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_splitkv_fp8(out, lse, dev.q, kc, vc, w.k_scale, w.v_scale, dev.block_tables,
                                 dev.seq_lens, w.scale, num_splits=Pu, workspace=ws,
                                 status=dev.status)
        assert_close(bf16_dev_to_f64(out), ref, f"{name} P={Pu}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"{name} P={Pu}")
    assert dev.status_value() == 0


@pytest.mark.parametrize("name", ["qwen2.5-7b-bs16-fp8", "qwen3-0.6b-B256-fp8", "long-B2-L32768-fp8"])
def test_fp8_step_full_size(name):
    """pa_decode_step_fp8: the fused quantising write leaves both pools byte for
    byte as the oracle's pa_cache_write_fp8 does, and the output equals the two
    calls (write, then decode) bit for bit and the oracle within tolerance,
    at auto P and unsplit."""
    w = W.WORKLOADS[name]()
    kc8, vc8 = w.k_cache8.copy(), w.v_cache8.copy()
    oracle.cache_write_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, w.k_scale, w.v_scale)
    ref, ref_lse = oracle.decode_fp8(w.q, kc8, vc8, w.block_tables, w.seq_lens, w.scale,
                                     w.k_scale, w.v_scale)
    dev = Dev(w)
    for P in (0, 1):
        Pu = P or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, Pu)),
                         dtype=torch.uint8, device="cuda")
        outs = []
        for fused in (True, False):
            kc, vc = _fp8_dev(w)
            out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
            if fused:
                pa.pa_decode_step_fp8(out, lse, dev.q, dev.k_new, dev.v_new, dev.slot_mapping, kc, vc,
                                      w.k_scale, w.v_scale, dev.block_tables, dev.seq_lens, w.scale,
                                      num_splits=Pu, workspace=ws, status=dev.status)
            else:
                pa.pa_cache_write_fp8(dev.k_new, dev.v_new, dev.slot_mapping, kc, vc, w.k_scale,
                                      w.v_scale, status=dev.status)
                pa.pa_decode_splitkv_fp8(out, lse, dev.q, kc, vc, w.k_scale, w.v_scale,
                                         dev.block_tables, dev.seq_lens, w.scale, num_splits=Pu,
                                         workspace=ws, status=dev.status)
            assert np.array_equal(kc.cpu().numpy(), kc8) and np.array_equal(vc.cpu().numpy(), vc8)
            outs.append((out, lse))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
        assert_close(bf16_dev_to_f64(outs[0][0]), ref, f"{name} fused P={Pu}")
        assert_lse_close(outs[0][1].cpu().double().numpy(), ref_lse, f"{name} fused P={Pu}")
    assert dev.status_value() == 0


def test_fp8_step_slots():
    """The fused FP8 write skips a negative slot and refuses (PA_STATUS_BAD_SLOT,
    nothing written) a slot that is not position L - 1 of its sequence; the
    other sequences' rows are written and attended as the oracle's."""
    lens = (40, 17, 100)
    w = W.with_fp8_pools(W.make_workload("f8s", B=3, Hq=16, Hkv=8, D=128, block_size=16,
                                         seq_lens=list(lens), num_blocks=20, seed=77))
    slots = w.slot_mapping.copy()
    slots[1] = -1
    dev = Dev(w)
    kc, vc = _fp8_dev(w)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    pa.pa_decode_step_fp8(out, None, dev.q, dev.k_new, dev.v_new, torch.from_numpy(slots).cuda(),
                          kc, vc, w.k_scale, w.v_scale, dev.block_tables, dev.seq_lens, w.scale,
                          num_splits=1, status=dev.status)
    kc8, vc8 = w.k_cache8.copy(), w.v_cache8.copy()
    oracle.cache_write_fp8(w.k_new, w.v_new, slots, kc8, vc8, w.k_scale, w.v_scale)
    assert np.array_equal(kc.cpu().numpy(), kc8) and np.array_equal(vc.cpu().numpy(), vc8)
    ref, _ = oracle.decode_fp8(w.q, kc8, vc8, w.block_tables, w.seq_lens, w.scale, w.k_scale,
                               w.v_scale)
    assert_close(bf16_dev_to_f64(out), ref, "fp8 step, one slot skipped")
    assert dev.status_value() == 0
    # sequence 2's slot moved to position 0 of sequence 0: not written, flagged
    bad = w.slot_mapping.copy()
    bad[2] = w.block_tables[0, 0] * 16
    kc, vc = _fp8_dev(w)
    pa.pa_decode_step_fp8(out, None, dev.q, dev.k_new, dev.v_new, torch.from_numpy(bad).cuda(),
                          kc, vc, w.k_scale, w.v_scale, dev.block_tables, dev.seq_lens, w.scale,
                          num_splits=1, status=dev.status)
    assert dev.status_value() & pa.PA_STATUS_BAD_SLOT
    written = bad.copy()
    written[2] = -1
    kc8, vc8 = w.k_cache8.copy(), w.v_cache8.copy()
    oracle.cache_write_fp8(w.k_new, w.v_new, written, kc8, vc8, w.k_scale, w.v_scale)
    assert np.array_equal(kc.cpu().numpy(), kc8) and np.array_equal(vc.cpu().numpy(), vc8)


# ------------------------------------------------ cascade decode (shared prefix)
CASCADE = [
    # (Hq, Hkv, bs, lens, shared prefix blocks)
    (16, 8, 16, (200, 129, 300, 150), 8),           # Qwen3-like, G = 2
    (28, 4, 16, (300, 257, 1000), 4),               # G = 7: one sequence per CTA column group
    (12, 2, 16, (70, 100, 33), 2),                  # G = 6
    (32, 2, 16, (129, 300), 3),                     # G = 16
    (16, 4, 256, (300, 513), 1),                    # 256-token pages
    (4, 2, 16, tuple(range(40, 80)), 2),            # 40 sequences: several query groups
]


@pytest.mark.parametrize("mode", ["always", "auto"])
@pytest.mark.parametrize("case", CASCADE, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-bs{c[2]}-B{len(c[3])}")
def test_cascade_matches_oracle(case, mode, cascade_mode):
    """The cascade (forced) and the automatic choice, which for these short
    prefixes is plain split decode."""
    cascade_mode(mode)
    Hq, Hkv, bs, lens, npre = case
    nb = sum((L + bs - 1) // bs for L in lens) + 5
    w = W.make_workload("casc", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, block_size=bs, seq_lens=list(lens),
                        num_blocks=nb, seed=npre + len(lens), shared_prefix_blocks=npre,
                        poison_unused=True, write_new=False)
    ref, ref_lse = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    ws = torch.zeros(max(1, pa.pa_cascade_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, npre, w.max_blocks,
                                                          w.block_size)), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    pa.pa_decode_cascade(out, lse, dev.q, dev.k_cache, dev.v_cache, npre, dev.block_tables,
                         dev.seq_lens, w.scale, workspace=ws, status=dev.status)
    assert_close(bf16_dev_to_f64(out), ref, "cascade")
    assert_lse_close(lse.cpu().double().numpy(), ref_lse, "cascade")
    assert dev.status_value() == 0


@pytest.mark.parametrize("mode", ["always", "auto"])
def test_cascade_full_size_qwen3(mode, cascade_mode):
    """The Qwen3 batch (256 sequences, 8 shared prefix blocks) after this step's
    write, through the cascade and through the automatic choice (plain split
    decode: these 8 blocks are read from L2 faster than the cascade's launches)."""
    cascade_mode(mode)
    w = W.WORKLOADS["qwen3-0.6b-B256-cascade"]()
    assert pa.pa_cascade_pays(w.B, w.Hkv, w.D, w.cascade_blocks, w.block_size) == (mode == "always")
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    ws = torch.zeros(pa.pa_cascade_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.cascade_blocks,
                                                   w.max_blocks, w.block_size),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    pa.pa_decode_cascade(out, lse, dev.q, dev.k_cache, dev.v_cache, w.cascade_blocks,
                         dev.block_tables, dev.seq_lens, w.scale, workspace=ws, status=dev.status)
    assert_close(bf16_dev_to_f64(out), ref, "cascade qwen3")
    assert_lse_close(lse.cpu().double().numpy(), ref_lse, "cascade qwen3")
    assert dev.status_value() == 0


@pytest.mark.parametrize("name,npre,pays", [("qwen3-0.6b-B256-prefix2048", 128, True),
                                            ("qwen3-0.6b-B8-prefix16384", 1024, True),
                                            ("qwen3-0.6b-B4-prefix65536", 4096, True)])
@pytest.mark.parametrize("cascade", [True, False])
def test_long_shared_prefix_full_size(name, npre, pays, cascade, cascade_mode):
    """Qwen3-shaped sequences behind one long shared prefix (256 behind 2048
    tokens, 8 behind 16384, 4 behind 65536), after this step's write: the
    cascade (prefix once for the whole batch, then each sequence's own
    blocks, then the merge: a combine kernel after the 256 unsplit suffixes,
    inside the split suffix pass for the others; forced where the automatic
    choice is plain decode) and the plain fused step, every row against the
    oracle's plain decode."""
    w = W.WORKLOADS[name]()
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    if cascade:
        cascade_mode("auto")
        assert bool(pa.pa_cascade_pays(w.B, w.Hkv, w.D, npre, w.block_size)) == pays  # the automatic choice
        if not pays:
            cascade_mode("always")
        dev.write()
        ws = torch.zeros(pa.pa_cascade_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, npre, w.max_blocks,
                                                       w.block_size), dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_cascade(out, lse, dev.q, dev.k_cache, dev.v_cache, npre, dev.block_tables,
                             dev.seq_lens, w.scale, workspace=ws, status=dev.status)
    else:
        out, lse, _ = dev.step(0)
    assert_close(bf16_dev_to_f64(out), ref, f"long prefix cascade={cascade}")
    assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"long prefix cascade={cascade}")
    assert dev.status_value() == 0


# ------------------------------------------------ a wait that nothing completes
def _preset_counters(w, P, value):
    """Split-KV workspace whose merge counters (its last region) all hold `value`."""
    ws = torch.zeros(pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P), dtype=torch.uint8,
                     device="cuda")
    rows = w.B * w.Hq * P
    rnd = lambda x: (x + 255) // 256 * 256                         # noqa: E731
    counters = rnd(rows * w.D * 4) + rnd(rows * 4)
    ws[counters:].view(torch.int32).fill_(value)
    return ws


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_merge_wait_times_out_and_the_context_survives(kernel, use_kernel, merge_path):
    """The grid-wide split merge waits for all P partitions to arrive; with the
    workspace's arrival counters preset far below zero that count is never
    reached.  Every CTA gives up after about a second, sets PA_STATUS_TIMEOUT
    and returns (the wait comes after all of the CTA's copies and MMAs have
    completed); the host reads the status and the next call is correct."""
    import time
    use_kernel(kernel)
    merge_path("grid")
    w = _small(28 if kernel == "tensor_core" else 8, 4, 128, 16, (1000,), seed=3)
    dev = Dev(w)
    dev.write()
    P = 4
    ws = _preset_counters(w, P, -(1 << 30))
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                         dev.seq_lens, w.scale, num_splits=P, workspace=ws, status=dev.status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert dev.status_value() & pa.PA_STATUS_TIMEOUT
    assert elapsed < 30, f"timed-out wait took {elapsed:.1f} s"
    dev.status.zero_()
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    so, sl, _ = dev.splitkv(P)
    assert_close(bf16_dev_to_f64(so), ref, f"after timeout {kernel}")
    assert dev.status_value() == 0


# ------------------------------------------- split merge: cluster and grid paths
MERGE_CASES = [
    # (Hq, Hkv, bs, lens)
    (28, 4, 16, (1000, 300, 1, 17)),        # G = 7, HC = 4; short sequences: empty partitions
    (16, 8, 16, (700, 129)),                # G = 2, HC = 8
    (48, 2, 16, (900, 65)),                 # G = 24: one head per CTA, 32 columns
    (16, 4, 256, (2000, 513, 2)),           # pages
]


@pytest.mark.parametrize("path", ["cluster", "grid"])
@pytest.mark.parametrize("case", MERGE_CASES, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-bs{c[2]}")
def test_split_merge_paths(case, path, merge_path):
    """pa_decode_splitkv and pa_decode_step at P = 2 .. 17 through either merge
    (P <= 16: one cluster per (sequence, head group) by default; 17: always the
    grid-wide merge), element by element against the oracle."""
    merge_path(path)
    Hq, Hkv, bs, lens = case
    w = _small(Hq, Hkv, 128, bs, lens, seed=sum(lens), poison_unused=True)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (2, 3, 8, 9, 16, 17):
        so, sl, _ = dev.splitkv(P)
        assert_close(bf16_dev_to_f64(so), ref, f"splitkv P={P} {path}")
        assert_lse_close(sl.cpu().double().numpy(), ref_lse, f"splitkv P={P} {path}")
    dev2 = Dev(w)
    for P in (4, 16):
        so, sl, _ = dev2.step(P)
        assert_close(bf16_dev_to_f64(so), ref, f"step P={P} {path}")
    assert dev.status_value() == 0 and dev2.status_value() == 0


@pytest.mark.parametrize("P", [2, 4, 9, 16])
def test_cluster_merge_leaves_the_counters_alone(P, merge_path):
    """With P <= 16 the partitions merge inside their cluster: the workspace's
    grid-merge counters are neither read nor written.  Preset far below zero
    (which makes the grid-wide merge time out), they do not delay or disturb
    the call, which shows the cluster path ran."""
    import time
    merge_path("cluster")
    w = _small(28, 4, 128, 16, (1000, 37), seed=P)
    dev = Dev(w)
    dev.write()
    dev.splitkv(P)                      # loads the kernel and sizes the cluster once
    ws = _preset_counters(w, P, -(1 << 30))
    before = ws.clone()
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    pa.pa_decode_splitkv(out, None, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                         dev.seq_lens, w.scale, num_splits=P, workspace=ws, status=dev.status)
    torch.cuda.synchronize()
    assert time.time() - t0 < 0.5
    assert dev.status_value() == 0
    rows = w.B * w.Hq * P
    tail = (rows * w.D * 4 + 255) // 256 * 256 + (rows * 4 + 255) // 256 * 256
    assert torch.equal(ws[tail:], before[tail:])
    kc, vc = oracle_after_write(w)
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    assert_close(bf16_dev_to_f64(out), ref, f"cluster P={P}")


@pytest.mark.parametrize("path", ["cluster", "grid"])
def test_split_merge_paths_mq_and_fp8(path, merge_path):
    """Multi-query (2 query groups per head group) and FP8 pools through either merge."""
    merge_path(path)
    w = W.make_workload("mq", B=3, Hq=28, Hkv=4, D=128, block_size=16, seq_lens=[900, 40, 3],
                        num_blocks=70, seed=12, poison_unused=True, q_len=4)
    kc, vc = oracle_after_write(w)
    ref, ref_lse = oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dev = Dev(w)
    dev.write()
    for P in (3, 16):
        out, lse, _ = dev.mq(P)
        assert_close(bf16_dev_to_f64(out), ref, f"mq P={P} {path}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"mq P={P} {path}")
    w = W.with_fp8_pools(W.make_workload("f8", B=2, Hq=28, Hkv=4, D=128, block_size=16,
                                         seq_lens=[1100, 9], num_blocks=80, seed=13,
                                         poison_unused=True, write_new=False))
    ref, ref_lse = oracle.decode_fp8(w.q, w.k_cache8, w.v_cache8, w.block_tables, w.seq_lens,
                                     w.scale, w.k_scale, w.v_scale)
    dev = Dev(w)
    k8, v8 = _fp8_dev(w)
    for P in (5, 16):
        ws = torch.zeros(pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_splitkv_fp8(out, lse, dev.q, k8, v8, w.k_scale, w.v_scale, dev.block_tables,
                                 dev.seq_lens, w.scale, num_splits=P, workspace=ws,
                                 status=dev.status)
        assert_close(bf16_dev_to_f64(out), ref, f"fp8 P={P} {path}")
        assert_lse_close(lse.cpu().double().numpy(), ref_lse, f"fp8 P={P} {path}")
    assert dev.status_value() == 0


# ------------------------------------- programmatic dependent launch: chained calls
@pytest.mark.parametrize("path", ["cluster", "grid"])
@pytest.mark.parametrize("graph", [False, True])
def test_chained_steps_see_the_previous_output(path, graph, merge_path):
    """The tensor-core kernel is launched with programmatic stream serialization,
    so a launch may become resident while the previous one finishes.  Chain
    eight calls whose queries are the previous call's output (a step's own
    fused write first), eagerly and replayed from a CUDA graph: each link must
    equal the oracle applied to the previous link's result, so no call may read
    its inputs before the previous kernel has written them."""
    merge_path(path)
    w = W.make_workload("chain", B=3, Hq=28, Hkv=4, D=128, block_size=16,
                        seq_lens=[300, 17, 129], num_blocks=40, seed=21)
    dev = Dev(w)
    P, n = 4, 8
    ws = [torch.zeros(pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P), dtype=torch.uint8,
                      device="cuda") for _ in range(n)]
    outs = [torch.full((w.B, w.Hq, w.D), 1e4, dtype=torch.bfloat16, device="cuda")
            for _ in range(n)]

    def chain():
        pa.pa_decode_step(outs[0], None, dev.q, dev.k_new, dev.v_new, dev.slot_mapping,
                          dev.k_cache, dev.v_cache, dev.block_tables, dev.seq_lens, w.scale,
                          num_splits=P, workspace=ws[0], status=dev.status)
        for i in range(1, n):
            pa.pa_decode_splitkv(outs[i], None, outs[i - 1], dev.k_cache, dev.v_cache,
                                 dev.block_tables, dev.seq_lens, w.scale, num_splits=P,
                                 workspace=ws[i], status=dev.status)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            chain()                                   # warm-up: loads the kernels
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for o in outs:
            o.fill_(1e4)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain()
        for o in outs:
            o.fill_(1e4)
        torch.cuda.synchronize()
        g.replay()
    else:
        chain()
    torch.cuda.synchronize()
    assert dev.status_value() == 0
    kc, vc = oracle_after_write(w)
    q = w.q
    for i in range(n):
        ref, _ = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, w.scale)
        got = bf16_dev_to_f64(outs[i])
        assert_close(got, ref, f"link {i} ({path}, graph={graph})")
        q = outs[i].view(torch.int16).cpu().numpy().view(np.uint16)   # the next link's queries
