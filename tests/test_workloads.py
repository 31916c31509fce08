"""The seeded input generators (paged_kv_decode_cache_gb300/workloads.py) on CPU:
the properties the input recipe states — reproducible bytes, block tables
that give every sequence its own scattered blocks (bar a shared prefix),
slots at each sequence's last positions, never-read rows poisoned, and the
FP8 variant's codes and scales.  No attention arithmetic is involved."""
import math

import numpy as np
import pytest
import torch

from paged_kv_decode_cache_gb300 import workloads as W


def _small(**kw):
    args = dict(B=5, Hq=8, Hkv=2, D=64, block_size=16, seq_lens=[1, 16, 17, 100, 33],
                num_blocks=40, seed=3)
    args.update(kw)
    return W.make_workload("t", **args)


def test_same_seed_same_bytes_other_seed_other_bytes():
    a, b, c = _small(), _small(), _small(seed=4)
    for f in ("q", "k_cache", "v_cache", "k_new", "v_new", "block_tables", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not np.array_equal(a.k_cache, c.k_cache)
    assert not np.array_equal(a.block_tables, c.block_tables)


def test_tables_give_each_sequence_its_own_blocks():
    w = _small()
    used = []
    for b, L in enumerate(w.seq_lens):
        nb = (int(L) + w.block_size - 1) // w.block_size
        row = w.block_tables[b]
        assert (row[:nb] >= 0).all() and (row[:nb] < w.num_blocks).all()
        assert (row[nb:] == -1).all()
        used.extend(row[:nb].tolist())
    assert len(used) == len(set(used))                  # no block in two sequences


def test_shared_prefix_blocks_are_the_same_physical_blocks():
    w = _small(seq_lens=[40, 70, 33], B=3, shared_prefix_blocks=2, write_new=False)
    assert (w.block_tables[:, :2] == w.block_tables[0, :2]).all()
    rest = [w.block_tables[b, 2:(int(L) + 15) // 16].tolist() for b, L in enumerate(w.seq_lens)]
    flat = sum(rest, [])
    assert len(flat) == len(set(flat)) and not set(flat) & set(w.block_tables[0, :2].tolist())


@pytest.mark.parametrize("q_len", [1, 4])
def test_slots_are_each_sequence_last_positions(q_len):
    w = _small(q_len=q_len, seq_lens=[1, 16, 17, 100, 33])
    assert w.slot_mapping.shape == (w.B * q_len,)
    for b, L in enumerate(w.seq_lens):
        for j in range(q_len):
            t = int(L) - q_len + j
            s = w.slot_mapping[b * q_len + j]
            if t < 0:
                assert s == -1                           # a position before the sequence starts
            else:
                assert s == w.block_tables[b, t // 16] * 16 + t % 16
    live = w.slot_mapping[w.slot_mapping >= 0]
    assert len(live) == len(set(live.tolist()))
    assert w.q.shape == ((w.B, w.Hq, w.D) if q_len == 1 else (w.B, q_len, w.Hq, w.D))


def test_poison_marks_exactly_the_rows_attention_never_reads():
    w = _small(poison_unused=True)
    live = np.zeros((w.num_blocks, w.block_size), bool)
    for b, L in enumerate(w.seq_lens):
        for t in range(int(L)):
            live[w.block_tables[b, t // 16], t % 16] = True
    nan = W.BF16_NAN
    assert (w.k_cache[~live] == nan).all() and (w.v_cache[~live] == nan).all()
    assert not (w.k_cache[live] == nan).any() and not (w.v_cache[live] == nan).any()


def test_bf16_inputs_are_rounded_standard_normals():
    w = _small()
    x = torch.from_numpy(w.k_cache.view(np.int16)).view(torch.bfloat16).float()
    assert torch.isfinite(x).all()
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05


def test_7b_layer_shape_and_byte_count():
    w = W.WORKLOADS["qwen2.5-7b-bs16"]()
    assert (w.B, w.Hq, w.Hkv, w.D, w.block_size) == (8, 28, 4, 128, 16)
    assert (w.seq_lens == 4096).all()
    assert w.scale == np.float32(1 / math.sqrt(128))
    assert w.kv_bytes() == 8 * 4096 * 2 * 4 * 128 * 2          # K + V, bf16
    assert w.qo_bytes() == 2 * 8 * 28 * 128 * 2


def test_fp8_variant_codes_and_scales():
    w = W.with_fp8_pools(_small())
    for bits, codes, scale in ((w.k_cache, w.k_cache8, w.k_scale), (w.v_cache, w.v_cache8, w.v_scale)):
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
        assert scale == pytest.approx(float(x.abs().max()) / 448.0, rel=1e-6)
        back = torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * scale
        err = (back - x).abs()
        # e4m3 keeps 3 mantissa bits: half an ulp is 2^-4 relative; below 2^-6 the
        # codes are subnormal with an absolute step of 2^-9 (times the scale)
        assert bool((err <= x.abs() * 2.0 ** -4 + scale * 2.0 ** -10 + 1e-12).all())
    assert w.name.endswith("-fp8") and w.fp8


def test_unique_bytes_count_a_shared_prefix_once():
    """Unique KV bytes: the prefix blocks every sequence shares count once; with
    no sharing they equal the logical bytes."""
    w = W.make_workload("u", B=3, Hq=4, Hkv=2, D=16, block_size=16, seq_lens=[40, 33, 17],
                        num_blocks=12, seed=1, shared_prefix_blocks=1, write_new=False)
    row = 2 * w.Hkv * w.D * 2
    assert w.kv_bytes() == (40 + 33 + 17) * row
    assert w.unique_kv_bytes() == (16 + (40 - 16) + (33 - 16) + (17 - 16)) * row
    w = W.make_workload("u", B=2, Hq=4, Hkv=2, D=16, block_size=16, seq_lens=[40, 5],
                        num_blocks=6, seed=1, write_new=False)
    assert w.unique_kv_bytes() == w.kv_bytes()
