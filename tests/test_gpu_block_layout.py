"""The write/read kernel at every launch geometry, at sizes the oracle checks in full.

The launch picks the row slice per CTA (32, 128 or 256 bytes: 1, 4 or 8 compute warps
of 32 bytes each) and the stage length from the shape and the GPU; the wide slices are
picked on their own only for shapes large enough to fill the GPU.  A test hook
(sdm_test_force_write_read_layout) forces them here, so that small shapes run the same
kernel instances as the full-size workloads: parity with the oracle, chunk-size
independence, bitwise repeatability, and the same bits for every slice and stage length
(the per-element arithmetic and its summation order depend on W and R only).
"""

import pytest
import torch

import sdm_inputs
from sdm_inputs import CONFIGS
from sdm_testlib import compare_stream, gpu_write_read

pytestmark = pytest.mark.gpu


@pytest.fixture
def layout():
    import gated_delta_rule_factor_gb300 as sdm

    def force(slice_bytes, stage_tokens=0):
        sdm.test_force_write_read_layout(slice_bytes, stage_tokens)
    yield force
    sdm.test_force_write_read_layout(0, 0)


VARIANTS = {
    "tiny": dict(),
    "w64_r64": dict(W=64, R=64, T=40),
    "w48_r64_ragged": dict(W=48, R=64, T=37, chunk_size=5),
    "w128_r96": dict(factor_dims=(64, 64), W=128, R=96, T=40, d_v=64),
    "w3_r5": dict(W=3, R=5, T=30),
    "one_write_one_read": dict(W=1, R=1),
    "bf16_bank": dict(act_dtype="bf16", bank_dtype="bf16", W=64, R=32, T=40, d_v=128),
    "f32_acts_bf16_bank": dict(bank_dtype="bf16", d_v=128, T=32),
    "bf16_acts": dict(act_dtype="bf16", d_v=96, W=24, R=40, T=40),
    "chunk_1": dict(T=40, chunk_size=1, W=32, R=32),
    "every_slot": dict(factor_dims=(4, 4), W=16, R=16, T=24),
    "three_factors": dict(factor_dims=(8, 8, 8), d_sub=16, W=16, R=12),
    "many_streams": dict(B=3, H=2, T=50, W=64, R=64),
    "long_head": dict(d_v=2048, T=24, W=64, R=64),
    "partial_last_slice": dict(d_v=40, T=30, W=64, R=64),
    "partial_last_slice_bf16": dict(d_v=72, bank_dtype="bf16", act_dtype="bf16", T=30),
}


@pytest.mark.parametrize("slice_bytes", [128, 256])
@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_wide_slices_match_oracle(layout, name, slice_bytes):
    kw = dict(VARIANTS[name])
    chunk = kw.pop("chunk_size", None)
    cfg = CONFIGS["tiny"].replace(**kw)
    layout(slice_bytes)
    d = sdm_inputs.make_inputs(cfg)
    gpu = gpu_write_read(cfg, d, chunk_size=chunk)
    res = [compare_stream(cfg, d, gpu, b, h) for b in range(cfg.B) for h in range(cfg.H)]
    assert sum(r["near_ties"] for r in res) <= 1, res


@pytest.mark.parametrize("slice_bytes", [32, 128, 256])
def test_chunk_size_changes_nothing(layout, slice_bytes):
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=200)
    layout(slice_bytes)
    d = sdm_inputs.make_inputs(cfg)
    ref = gpu_write_read(cfg, d, chunk_size=64)
    for c in (1, 2, 3, 17, 128, 256):
        out = gpu_write_read(cfg, d, chunk_size=c)
        for k in ref:
            assert torch.equal(ref[k], out[k]), (c, k)


def test_bitwise_repeatable_at_every_slice(layout):
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=120, d_v=256)
    d = sdm_inputs.make_inputs(cfg)
    for sb in (32, 128, 256):
        layout(sb)
        first = gpu_write_read(cfg, d)
        for _ in range(2):
            out = gpu_write_read(cfg, d)
            for k in first:
                assert torch.equal(first[k], out[k]), (sb, k)


@pytest.mark.parametrize("bank_dtype", ["f32", "bf16"])
def test_results_do_not_depend_on_the_slice_or_the_stage_length(layout, bank_dtype):
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=60, d_v=256, bank_dtype=bank_dtype)
    d = sdm_inputs.make_inputs(cfg)
    layout(0)
    ref = gpu_write_read(cfg, d)
    for sb, g in ((32, 0), (128, 0), (256, 0), (128, 1), (256, 2), (32, 5)):
        layout(sb, g)
        out = gpu_write_read(cfg, d)
        for k in ref:
            assert torch.equal(ref[k], out[k]), (sb, g, k)
