"""The C-ABI library builds, loads and exports every function include/pa.h
declares; host-side logic (split policy, workspace sizing, argument checks
that reject before any CUDA call) behaves as documented.  No GPU needed."""
import ctypes
import subprocess

import numpy as np
import pytest
import torch

from paged_kv_decode_cache_gb300 import build as B
from paged_kv_decode_cache_gb300 import pa


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pa.lib()


def test_header_declares_the_boundary():
    names = set(pa.header_functions())
    for required in ("pa_cache_write", "pa_decode", "pa_decode_splitkv", "pa_combine",
                     "pa_decode_partial", "pa_choose_num_splits", "pa_splitkv_workspace_bytes",
                     "pa_strerror"):
        assert required in names


def test_every_declared_function_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in pa.header_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in pa.header_functions():
        assert isinstance(getattr(lib, n), ctypes._CFuncPtr)


def test_binding_covers_the_header():
    assert set(pa.header_functions()) == set(pa._SIGNATURES)


def test_version_and_strerror(lib):
    assert pa.pa_version() >= 100
    for code in (pa.PA_OK, pa.PA_EINVAL, pa.PA_EUNSUPPORTED, pa.PA_EWORKSPACE, pa.PA_ECUDA):
        assert pa.pa_strerror(code) and pa.pa_strerror(code) != "unknown error code"
    assert pa.pa_strerror(-99) == "unknown error code"


# (B, Hq, Hkv, D, max_blocks, bs, sms); CTAs per SM: 1 for the tensor-core
# kernel (D = 128, G >= 4), 2 for the CUDA-core kernel.
SPLIT_CASES = [
    (8, 28, 4, 128, 256, 16, 152), (1, 28, 4, 128, 2048, 16, 152), (2, 28, 4, 128, 2048, 16, 152),
    (256, 16, 8, 128, 128, 16, 152), (8, 12, 2, 128, 128, 16, 152), (1, 12, 2, 128, 128, 16, 152),
    (8, 28, 4, 128, 16, 256, 152), (4, 4, 2, 64, 7, 16, 152), (1, 1, 1, 64, 1, 16, 152),
    (3, 2, 1, 128, 1000, 16, 132),
]


def _tc_heads_per_cta(G, Hkv):
    """KV heads per CTA of the tensor-core kernel (mirrors the library's rule)."""
    hc = 1
    while hc < 8 and Hkv % (hc * 2) == 0:
        hc *= 2
    if G > 16:      # more than 16 columns: one KV head per CTA
        hc = 1
    while True:
        gp = 1
        while gp < G:
            gp *= 2
        gp = max(gp, 16 // hc)
        if gp * hc <= 64:
            return hc
        hc //= 2


def _ctas_per_sm(Hq, Hkv, D):
    return 1 if D == 128 else 2


def _units(B, Hq, Hkv, D):
    return B * (Hkv // _tc_heads_per_cta(Hq // Hkv, Hkv)) if D == 128 else B * Hkv


@pytest.mark.parametrize("B,Hq,Hkv,D,mb,bs,sms", SPLIT_CASES)
def test_split_policy(lib, use_kernel, B, Hq, Hkv, D, mb, bs, sms):
    use_kernel("auto")
    P = pa.pa_choose_num_splits(B, Hq, Hkv, D, mb, bs, sms)
    lmax = mb * bs
    slots = _ctas_per_sm(Hq, Hkv, D) * sms
    assert 1 <= P <= 256
    chunk = pa.pa_partition_tokens(mb, bs, P)
    assert chunk % 16 == 0 and chunk * P >= lmax and chunk * (P - 1) < lmax  # no empty tail split
    units = _units(B, Hq, Hkv, D)
    if P > 1 and units <= slots:
        assert units * P <= slots              # one wave of resident CTAs
        assert chunk >= 16 * 2 or chunk * P >= lmax
        tiles = (lmax + 15) // 16
        assert P <= 32 or -(-tiles // 4) > 32  # the wider merge only where 4-tile partitions need it
    if units > slots:   # waves: partitions of about 48 tiles, without empty tails
        tiles = (lmax + 15) // 16
        p0 = min(-(-tiles // 48), -(-tiles // 2))
        assert P == -(-lmax // pa.pa_partition_tokens(mb, bs, max(1, p0)))


def test_multi_wave_batches_split_into_48_tile_partitions(lib, use_kernel):
    use_kernel("auto")
    # the Qwen3 batch: 256 sequences of up to 2048 tokens, 8 KV heads per CTA, 148 SMs
    assert pa.pa_choose_num_splits(256, 16, 8, 128, 128, 16, 148) == 3
    assert pa.pa_choose_num_splits(256, 16, 8, 128, 16, 16, 148) == 1      # 256 tokens: one partition
    assert pa.pa_choose_num_splits(148, 16, 8, 128, 128, 16, 148) == 1     # exactly one wave


def test_decode_launches(lib, use_kernel):
    use_kernel("auto")
    L = pa.pa_decode_launches
    assert L(8, 1, 28, 4, 128, 256, 16, 1, 148) == 1          # unsplit
    assert L(8, 1, 28, 4, 128, 256, 16, 0, 148) == 1          # split, one wave: merged in the launch
    assert L(1, 1, 28, 4, 128, 2048, 16, 0, 148) == 1
    assert L(256, 1, 16, 8, 128, 128, 16, 0, 148) == 2        # waves: partials, then the combine
    assert L(8, 1, 28, 4, 128, 4096, 16, 257, 148) == 2       # more partitions than a merge task holds
    assert L(8, 512, 12, 2, 128, 128, 16, 2, 148) == 2        # the prefill-shaped kernel
    assert L(0, 1, 28, 4, 128, 256, 16, 0, 148) == 0
    assert lib.pa_decode_launches(8, 1, 28, 5, 128, 256, 16, 0, 148) == pa.PA_EINVAL
    assert lib.pa_decode_launches(8, 1, 28, 4, 128, 256, 16, 0, 0) == pa.PA_EINVAL


def test_split_policy_properties_on_random_shapes(lib, use_kernel):
    """The split choice's rules on 300 seeded shapes: 1 <= P <= 256; no empty
    tail partition; partitions of at least 2 tiles; more than 32 partitions
    only where 4-tile partitions would already number more than 32; one wave
    of resident CTAs whenever the units alone fit."""
    use_kernel("auto")
    rng = np.random.default_rng(2024)
    for _ in range(300):
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 6, 7, 8]))
        B = int(rng.integers(1, 300))
        bs = int(rng.choice([16, 32, 256]))
        mb = int(rng.integers(1, 4096 // bs + 2))
        sms = int(rng.choice([132, 148, 152]))
        Hq = G * Hkv
        P = pa.pa_choose_num_splits(B, Hq, Hkv, 128, mb, bs, sms)
        lmax = mb * bs
        tiles = -(-lmax // 16)
        assert 1 <= P <= 256
        chunk = pa.pa_partition_tokens(mb, bs, P)
        assert chunk * P >= lmax and chunk * (P - 1) < lmax
        assert P == 1 or chunk >= 32
        assert P <= 32 or -(-tiles // 4) > 32
        units = _units(B, Hq, Hkv, 128)
        if units <= sms and P > 1:
            assert units * P <= sms


def test_split_policy_short_contexts(lib, use_kernel):
    use_kernel("auto")
    # the 7B layer at 256 tokens: partitions of 2 tiles (8 per sequence, 64 CTAs)
    assert pa.pa_choose_num_splits(8, 28, 4, 128, 16, 16, 152) == 8
    # one 2k-token sequence: 32 partitions of 4 tiles, not 64 of 2 (the wider merge)
    assert pa.pa_choose_num_splits(1, 12, 2, 128, 128, 16, 152) == 32
    # one 4k-token sequence: 4-tile partitions would already be 64, so 2-tile ones
    assert pa.pa_choose_num_splits(1, 28, 4, 128, 256, 16, 152) == 128


def test_cascade_launches(lib, use_kernel, cascade_mode):
    use_kernel("auto")
    cascade_mode("auto")
    C = pa.pa_cascade_launches
    # 256 sequences behind 8 shared blocks: no cascade; the plain split runs in
    # waves (P = 3): partials, then the combine
    assert C(256, 16, 8, 128, 8, 128, 16, 148) == 2
    # 256 behind 2048 tokens: prefix pass, unsplit suffix pass, combine
    assert C(256, 16, 8, 128, 128, 144, 16, 148) == 3
    # 8 behind 16384 tokens: the split suffix pass merges both passes' partials
    assert C(8, 16, 8, 128, 1024, 1040, 16, 148) == 2
    assert C(0, 16, 8, 128, 8, 128, 16, 148) == 0
    assert lib.pa_cascade_launches(8, 16, 8, 128, 128, 128, 16, 148) == pa.PA_EINVAL  # no own blocks
    assert lib.pa_cascade_launches(8, 16, 8, 128, 8, 128, 16, 0) == pa.PA_EINVAL
    cascade_mode("never")
    assert C(256, 16, 8, 128, 128, 144, 16, 148) == 2    # plain split in waves + combine
    assert C(8, 16, 8, 128, 1024, 1040, 16, 148) == 1    # plain split, merged in the launch


def test_split_policy_fills_small_batches(lib, use_kernel):
    use_kernel("auto")
    # one work unit (B=1, all 4 KV heads in one CTA) at 32k tokens: the split fills every SM
    P = pa.pa_choose_num_splits(1, 28, 4, 128, 2048, 16, 152)
    assert P >= 0.9 * 152
    # the CUDA-core kernel has one CTA per KV head and two CTAs per SM
    use_kernel("cuda_core")
    assert 4 * pa.pa_choose_num_splits(1, 28, 4, 128, 2048, 16, 152) >= 0.9 * 2 * 152


def test_kernel_override_rejects_what_it_cannot_run(lib, use_kernel):
    use_kernel("tensor_core")
    assert lib.pa_choose_num_splits(1, 8, 2, 64, 16, 16, 152) == pa.PA_EUNSUPPORTED   # D = 64
    use_kernel("cuda_core")
    assert lib.pa_choose_num_splits(1, 32, 2, 128, 16, 16, 152) == pa.PA_EUNSUPPORTED  # G = 16
    use_kernel("auto")
    assert lib.pa_choose_num_splits(1, 32, 2, 128, 16, 16, 152) >= 1                   # tensor cores
    assert lib.pa_choose_num_splits(1, 64, 2, 128, 16, 16, 152) >= 1                   # G = 32
    assert lib.pa_choose_num_splits(1, 66, 2, 128, 16, 16, 152) == pa.PA_EUNSUPPORTED  # G = 33


def test_partition_tokens(lib):
    assert pa.pa_partition_tokens(256, 16, 1) == 4096
    assert pa.pa_partition_tokens(256, 16, 9) == 464
    assert pa.pa_partition_tokens(7, 16, 3) == 48
    assert lib.pa_partition_tokens(0, 16, 1) == pa.PA_EINVAL


def test_workspace_bytes(lib):
    assert pa.pa_splitkv_workspace_bytes(8, 28, 128, 1) == 0
    n = pa.pa_splitkv_workspace_bytes(8, 28, 128, 9)
    rows = 8 * 28 * 9
    assert n >= rows * 128 * 4 + rows * 4 and n % 256 == 0


def _desc(nb=64, bs=16, hkv=2, d=64):
    return pa.CacheDesc(nb, bs, hkv, d)


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: these calls fail validation first


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), pa.PA_EINVAL),
    (dict(q=None), pa.PA_EINVAL),
    (dict(Hq=5), pa.PA_EINVAL),                 # Hq % Hkv != 0
    (dict(Hq=18), pa.PA_EUNSUPPORTED),          # G = 9 > 8 at D = 64
    (dict(Hq=66, desc=_desc(d=128)), pa.PA_EUNSUPPORTED),   # G = 33 > 32
    (dict(desc=_desc(d=96)), pa.PA_EUNSUPPORTED),
    (dict(desc=_desc(bs=8)), pa.PA_EUNSUPPORTED),
    (dict(desc=_desc(nb=0)), pa.PA_EINVAL),
    (dict(max_blocks=0), pa.PA_EINVAL),
    (dict(q=ctypes.c_void_p((1 << 20) + 2)), pa.PA_EINVAL),   # misaligned
    (dict(scale=float("nan")), pa.PA_EINVAL),
    (dict(B=70000), pa.PA_EUNSUPPORTED),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    a = dict(out=FAKE, lse=None, q=FAKE, k=FAKE, v=FAKE, desc=_desc(), bt=FAKE, max_blocks=7,
             sl=FAKE, B=4, Hq=4, scale=0.125, status=None, stream=None)
    a.update(kw)
    rc = lib.pa_decode(a["out"], a["lse"], a["q"], a["k"], a["v"], a["desc"], a["bt"],
                       a["max_blocks"], a["sl"], a["B"], a["Hq"], a["scale"], a["status"],
                       a["stream"])
    assert rc == code


def test_empty_batch_is_a_noop(lib):
    assert lib.pa_decode(FAKE, None, FAKE, FAKE, FAKE, _desc(), FAKE, 7, FAKE, 0, 4, 0.1,
                         None, None) == pa.PA_OK
    assert lib.pa_cache_write(FAKE, FAKE, FAKE, 0, FAKE, FAKE, _desc(), None, None) == pa.PA_OK


def test_splitkv_rejects_missing_workspace(lib):
    rc = lib.pa_decode_splitkv(FAKE, None, FAKE, FAKE, FAKE, _desc(), FAKE, 7, FAKE, 4, 4, 0.1,
                               4, None, 0, None, None)
    assert rc == pa.PA_EWORKSPACE
    rc = lib.pa_decode_splitkv(FAKE, None, FAKE, FAKE, FAKE, _desc(), FAKE, 7, FAKE, 4, 4, 0.1,
                               -1, None, 0, None, None)
    assert rc == pa.PA_EINVAL


def test_combine_and_write_reject_bad_arguments(lib):
    assert lib.pa_combine(FAKE, None, FAKE, FAKE, 2, 4, 0, 128, None) == pa.PA_EINVAL
    assert lib.pa_combine(FAKE, None, FAKE, FAKE, 2, 4, 3, 80, None) == pa.PA_EUNSUPPORTED
    assert lib.pa_cache_write(None, FAKE, FAKE, 3, FAKE, FAKE, _desc(), None, None) == pa.PA_EINVAL
    assert lib.pa_cache_write(FAKE, FAKE, FAKE, -1, FAKE, FAKE, _desc(), None, None) == pa.PA_EINVAL
    assert lib.pa_decode_partial(FAKE, FAKE, FAKE, FAKE, FAKE, _desc(), FAKE, 7, FAKE, 4, 4, 0.1,
                                 0, None, None) == pa.PA_EINVAL


def test_decode_step_rejects_bad_arguments(lib):
    d = _desc()
    args = lambda **kw: [kw.get(k, FAKE) for k in ("out",)] + [None] + [
        kw.get(k, FAKE) for k in ("q", "kn", "vn", "slots", "k", "v")]
    base = dict(out=FAKE, q=FAKE, kn=FAKE, vn=FAKE, slots=FAKE, k=FAKE, v=FAKE)
    for bad in ("kn", "vn", "slots"):
        a = dict(base, **{bad: None})
        rc = lib.pa_decode_step(a["out"], None, a["q"], a["kn"], a["vn"], a["slots"], a["k"], a["v"],
                                d, FAKE, 7, FAKE, 4, 4, 0.125, 1, None, 0, None, None)
        assert rc == pa.PA_EINVAL, bad
    rc = lib.pa_decode_step(FAKE, None, FAKE, ctypes.c_void_p((1 << 20) + 8), FAKE, FAKE, FAKE, FAKE,
                            d, FAKE, 7, FAKE, 4, 4, 0.125, 1, None, 0, None, None)
    assert rc == pa.PA_EINVAL   # misaligned k_new
    assert lib.pa_decode_step(None, None, None, None, None, None, None, None, d, None, 7, None, 0,
                              4, 0.125, 1, None, 0, None, None) == pa.PA_OK   # empty batch


def test_mq_split_policy(lib, use_kernel):
    use_kernel("auto")
    for args in ((8, 28, 4, 128, 256, 16, 152), (1, 28, 4, 128, 2048, 16, 152),
                 (256, 16, 8, 128, 128, 16, 152), (3, 12, 2, 128, 100, 16, 132)):
        B, Hq, Hkv, D, mb, bs, sms = args
        assert pa.pa_choose_num_splits_mq(B, 1, Hq, Hkv, D, mb, bs, sms) == \
            pa.pa_choose_num_splits(B, Hq, Hkv, D, mb, bs, sms)
    # 7B layer, 4 queries: 32 // 7 = 4 positions per CTA -> 28 columns, one KV head
    # per CTA -> 4 CTAs per sequence per split -> one wave of 152 SMs holds P = 4
    assert pa.pa_choose_num_splits_mq(8, 4, 28, 4, 128, 256, 16, 152) == 4
    # Qwen3 shape, 4 queries: all fit one CTA per 8 KV heads -> as q_len = 1 (256 units:
    # waves, partitions of 48 tiles)
    assert pa.pa_choose_num_splits_mq(256, 4, 16, 8, 128, 128, 16, 152) == 3
    # more query groups never give more splits
    prev = 10 ** 9
    for q_len in (1, 2, 3, 5, 8, 16, 64):
        P = pa.pa_choose_num_splits_mq(1, q_len, 12, 2, 128, 512, 16, 152)
        assert 1 <= P <= prev
        prev = P


def test_mq_rejects_what_it_cannot_run(lib, use_kernel):
    use_kernel("auto")
    assert lib.pa_choose_num_splits_mq(2, 2, 8, 2, 64, 16, 16, 152) == pa.PA_EUNSUPPORTED   # D = 64
    assert lib.pa_choose_num_splits_mq(2, 0, 8, 2, 128, 16, 16, 152) == pa.PA_EINVAL
    assert lib.pa_choose_num_splits_mq(2, 1, 8, 2, 64, 16, 16, 152) >= 1                    # decode
    use_kernel("cuda_core")
    assert lib.pa_choose_num_splits_mq(2, 2, 8, 2, 128, 16, 16, 152) == pa.PA_EUNSUPPORTED
    use_kernel("auto")
    d = _desc(d=128)
    for q_len in (0, -3, 70000):
        rc = lib.pa_decode_mq(FAKE, None, FAKE, q_len, FAKE, FAKE, d, FAKE, 7, FAKE, 4, 4, 0.1, 1,
                              None, 0, None, None)
        assert rc == pa.PA_EINVAL, q_len
    rc = lib.pa_decode_mq(FAKE, None, FAKE, 2, FAKE, FAKE, d, FAKE, 7, FAKE, 4, 4, 0.1, 3,
                          None, 0, None, None)
    assert rc == pa.PA_EWORKSPACE       # P > 1 without a workspace
    rc = lib.pa_decode_mq(FAKE, None, FAKE, 2, FAKE, FAKE, _desc(d=64), FAKE, 7, FAKE, 4, 4, 0.1, 1,
                          None, 0, None, None)
    assert rc == pa.PA_EUNSUPPORTED     # D = 64


def test_fp8_rejects_bad_arguments(lib, use_kernel):
    use_kernel("auto")
    d = _desc(d=128)
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert lib.pa_cache_write_fp8(FAKE, FAKE, FAKE, 3, FAKE, FAKE, d, ks, vs, None, None) == pa.PA_EINVAL
        assert lib.pa_decode_splitkv_fp8(FAKE, None, FAKE, FAKE, FAKE, d, ks, vs, FAKE, 7, FAKE, 4, 4,
                                         0.1, 1, None, 0, None, None) == pa.PA_EINVAL
    assert lib.pa_decode_splitkv_fp8(FAKE, None, FAKE, FAKE, FAKE, _desc(d=64), 1.0, 1.0, FAKE, 7,
                                     FAKE, 4, 4, 0.1, 1, None, 0, None, None) == pa.PA_EUNSUPPORTED
    assert lib.pa_decode_splitkv_fp8(FAKE, None, FAKE, FAKE, FAKE, d, 1.0, 1.0, FAKE, 7, FAKE, 4, 4,
                                     0.1, 3, None, 0, None, None) == pa.PA_EWORKSPACE
    use_kernel("cuda_core")
    assert lib.pa_decode_splitkv_fp8(FAKE, None, FAKE, FAKE, FAKE, d, 1.0, 1.0, FAKE, 7, FAKE, 4, 4,
                                     0.1, 1, None, 0, None, None) == pa.PA_EUNSUPPORTED
    assert lib.pa_cache_write_fp8(FAKE, FAKE, FAKE, 0, FAKE, FAKE, d, 1.0, 1.0, None, None) == pa.PA_OK


def test_cascade_rejects_bad_arguments(lib):
    d = _desc(d=128)
    for npre in (-1, 7, 9):   # max_blocks = 7
        rc = lib.pa_decode_cascade(FAKE, None, FAKE, FAKE, FAKE, d, npre, FAKE, 7, FAKE, 4, 4, 0.1,
                                   None, 0, None, None)
        assert rc == pa.PA_EINVAL, npre
    assert lib.pa_cascade_workspace_bytes(4, 4, 4, 128, 0, 7, 16) == 0
    assert lib.pa_cascade_workspace_bytes(4, 4, 4, 128, 7, 7, 16) == 0


def test_wrappers_run_on_their_tensors_device():
    """Every tensor wrapper checks that its tensors share one CUDA device (and
    runs there); the check itself needs no GPU."""
    one = pa._one_cuda_device
    assert one([torch.device("cpu")], "f") is None
    assert one([torch.device("cuda", 1), torch.device("cuda", 1), torch.device("cpu")], "f") == \
        torch.device("cuda", 1)
    with pytest.raises(ValueError, match="several devices"):
        one([torch.device("cuda", 0), torch.device("cuda", 1)], "f")
    for name in ("pa_cache_write", "pa_decode", "pa_decode_partial", "pa_combine",
                 "pa_decode_splitkv", "pa_decode_step", "pa_decode_mq", "pa_decode_cascade",
                 "pa_cache_write_fp8", "pa_decode_splitkv_fp8", "pa_decode_splitkv_noalloc"):
        assert getattr(pa, name).__wrapped__.__name__ == name


def test_options_set_get_and_reject(lib):
    opts = (pa.PA_OPT_DECODE_KERNEL, pa.PA_OPT_SPLIT_MERGE, pa.PA_OPT_PDL, pa.PA_OPT_CASCADE)
    prev = [pa.pa_get_option(o) for o in opts]
    try:
        for opt, values in ((pa.PA_OPT_DECODE_KERNEL, (0, 1, 2)), (pa.PA_OPT_SPLIT_MERGE, (0, 1)),
                            (pa.PA_OPT_PDL, (0, 1)), (pa.PA_OPT_CASCADE, (0, 1, 2))):
            for v in values:
                pa.pa_set_option(opt, v)
                assert pa.pa_get_option(opt) == v
            assert lib.pa_set_option(opt, max(values) + 1) == pa.PA_EINVAL
            assert lib.pa_set_option(opt, -1) == pa.PA_EINVAL
        assert lib.pa_set_option(4, 0) == pa.PA_EINVAL
        assert lib.pa_get_option(4) == pa.PA_EINVAL
        # the split policy follows the switch, not the environment
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, pa.PA_KERNEL_CUDA_CORE)
        assert lib.pa_choose_num_splits(1, 32, 2, 128, 16, 16, 152) == pa.PA_EUNSUPPORTED
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, pa.PA_KERNEL_AUTO)
        assert lib.pa_choose_num_splits(1, 32, 2, 128, 16, 16, 152) >= 1
    finally:
        for o, v in zip(opts, prev):
            pa.pa_set_option(o, v)


def test_options_start_from_the_environment_read_once(lib, tmp_path):
    """In a fresh process the switches start from PA_DECODE_KERNEL, PA_SPLIT_MERGE
    and PA_PDL; changing the environment afterwards changes nothing."""
    import os
    import sys
    code = (
        "import os, sys; sys.path.insert(0, %r)\n"
        "from paged_kv_decode_cache_gb300 import pa\n"
        "a = [pa.pa_get_option(o) for o in (0, 1, 2)]\n"
        "os.environ['PA_DECODE_KERNEL'] = 'tensor_core'; os.environ['PA_PDL'] = '1'\n"
        "b = [pa.pa_get_option(o) for o in (0, 1, 2)]\n"
        "print(a, b)\n" % os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    env = dict(os.environ, PA_DECODE_KERNEL="cuda_core", PA_SPLIT_MERGE="grid", PA_PDL="0")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True).stdout.strip()
    assert out == "[1, 1, 0] [1, 1, 0]"


@pytest.mark.parametrize("kw,code", [
    (dict(desc=_desc(d=0)), pa.PA_EINVAL),
    (dict(desc=_desc(d=-1)), pa.PA_EINVAL),
    (dict(desc=_desc(d=256)), pa.PA_EUNSUPPORTED),
    (dict(Hq=5), pa.PA_EINVAL),                 # Hq % Hkv != 0
    (dict(q=None), pa.PA_EINVAL),
    (dict(out=None), pa.PA_EINVAL),
    (dict(splits=-1), pa.PA_EINVAL),
    (dict(splits=70000), pa.PA_EUNSUPPORTED),
    (dict(B=-1), pa.PA_EINVAL),
])
def test_noalloc_rejects_bad_arguments_before_touching_its_array(lib, kw, code):
    """The allocation-free entry point checks its arguments exactly as
    pa_decode_splitkv does, before it looks up or clears its built-in array
    (no CUDA call is made here: this machine may have no GPU)."""
    a = dict(out=FAKE, q=FAKE, desc=_desc(), B=4, Hq=4, splits=4)
    a.update(kw)
    rc = lib.pa_decode_splitkv_noalloc(a["out"], None, a["q"], FAKE, FAKE, a["desc"], FAKE, 7, FAKE,
                                       a["B"], a["Hq"], 0.125, a["splits"], None, None)
    assert rc == code


def test_mq_split_policy_prefill_shape(lib, use_kernel):
    """Calls with more query columns per KV head than the decode kernel holds
    (q_len * G > 32) count one CTA per (sequence, KV head, tile of 128 / G
    positions); a partition never exceeds 2048 tiles of 16 tokens."""
    use_kernel("auto")
    # Qwen2.5-1.5B layer, 512-token chunk: 21 positions per tile -> 25 tiles per KV head
    assert pa.pa_choose_num_splits_mq(8, 512, 12, 2, 128, 128, 16, 152) == 1       # 400 CTAs
    assert pa.pa_choose_num_splits_mq(1, 512, 12, 2, 128, 128, 16, 152) == 3       # 50 CTAs
    # G = 7, 64 queries: 18 positions per tile -> 4 tiles
    assert pa.pa_choose_num_splits_mq(2, 64, 28, 4, 128, 256, 16, 152) == 4        # 32 CTAs x 4
    # a 64k-token table needs at least 2 partitions of at most 32768 tokens
    assert pa.pa_choose_num_splits_mq(64, 128, 8, 1, 128, 4096, 16, 152) >= 2


def test_cascade_runs_where_it_pays(lib, cascade_mode):
    """The automatic choice: the cascade when (B - 1) x the prefix's K/V bytes
    reach 256 MiB; the switch forces either path."""
    cascade_mode("auto")
    assert not pa.pa_cascade_pays(256, 8, 128, 8, 16)      # 8 blocks: 255 x 512 KiB = 128 MiB
    assert pa.pa_cascade_pays(256, 8, 128, 128, 16)        # 2048 tokens: 255 x 8 MiB
    assert pa.pa_cascade_pays(8, 8, 128, 1024, 16)         # 16384 tokens: 7 x 64 MiB
    assert pa.pa_cascade_pays(4, 8, 128, 4096, 16)         # 65536 tokens: 3 x 256 MiB
    assert not pa.pa_cascade_pays(2, 8, 128, 1024, 16)     # 16384 tokens read once more: 64 MiB
    assert not pa.pa_cascade_pays(1, 8, 128, 4096, 16)     # one sequence: nothing to share
    assert pa.pa_cascade_pays(9, 8, 128, 2048, 16)         # a 128 MiB prefix read 8 more times
    assert pa.pa_cascade_pays(3, 8, 128, 2048, 16)         # ... or 2 more times
    assert not pa.pa_cascade_pays(256, 8, 128, 0, 16)
    assert lib.pa_cascade_pays(0, 8, 128, 8, 16) == pa.PA_EINVAL
    cascade_mode("always")
    assert pa.pa_cascade_pays(256, 8, 128, 8, 16)
    cascade_mode("never")
    assert not pa.pa_cascade_pays(256, 8, 128, 128, 16)

