"""pa_decode_splitkv_noalloc: split-KV decode for callers that cannot allocate.

Some callers cannot call cudaMalloc (or any allocator) where they run decode,
so they cannot hand pa_decode_splitkv a workspace: this entry point keeps the
split's partial results in a device array built into the library instead.
The test calls it through the C ABI twice in a row, with different queries,
and checks each result against pa_decode_splitkv with a caller-allocated
workspace.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from gpu_util import Dev, assert_close, assert_lse_close, bf16_dev_to_f64
from paged_kv_decode_cache_gb300 import pa
from paged_kv_decode_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_decode_cache_gb300 import build
    build.build()


def _noalloc(dev, P):
    w = dev.w
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitkv_noalloc(out, lse, dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                                 dev.seq_lens, w.scale, num_splits=P, status=dev.status)
    return out, lse


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    w = W.qwen25_7b(16)
    dev = Dev(w)
    dev.write()
    P = pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
    assert P > 1
    assert pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P) <= pa.PA_NOALLOC_SCRATCH_BYTES
    ref1, ref1_lse, _ = dev.splitkv(P)
    got1, got1_lse = _noalloc(dev, P)
    # second call, different queries: the shared scratch must not leak the first call's data
    q2 = torch.flip(dev.q, dims=[1]).contiguous()
    dev.q = q2
    ref2, ref2_lse, _ = dev.splitkv(P)
    got2, got2_lse = _noalloc(dev, P)
    torch.cuda.synchronize()
    assert dev.status_value() == 0
    for got, gl, ref, rl, tag in ((got1, got1_lse, ref1, ref1_lse, "call 1"),
                                  (got2, got2_lse, ref2, ref2_lse, "call 2")):
        assert_close(bf16_dev_to_f64(got), bf16_dev_to_f64(ref), f"noalloc {tag}")
        assert_lse_close(gl.cpu().double().numpy(), rl.cpu().double().numpy(), f"noalloc {tag}")
    assert not torch.equal(got1, got2)


def test_noalloc_rejects_splits_beyond_the_builtin_array():
    w = W.make_workload("big", B=64, Hq=32, Hkv=4, D=128, block_size=16, seq_lens=[16] * 64,
                        num_blocks=80, max_blocks=1, seed=3, write_new=False)
    dev = Dev(w)
    P = 64
    assert pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P) > pa.PA_NOALLOC_SCRATCH_BYTES
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_splitkv_noalloc(out, None, dev.q, dev.k_cache, dev.v_cache,
                                     dev.block_tables, dev.seq_lens, w.scale, num_splits=P)
    assert e.value.code == pa.PA_EWORKSPACE


def test_noalloc_unsplit_call_equals_pa_decode():
    """num_splits = 1 does not use the built-in array: the result is pa_decode's, bit for bit."""
    w = W.make_workload("one", B=3, Hq=28, Hkv=4, D=128, block_size=16, seq_lens=[300, 17, 1],
                        num_blocks=30, seed=4)
    dev = Dev(w)
    dev.write()
    ref, ref_lse = dev.decode()
    got, got_lse = _noalloc(dev, 1)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse)
    assert dev.status_value() == 0

