"""The write/read kernel on 128-byte row slices (block-ordered token step) at small sizes.

The launch picks 128-byte slices on its own only when a shape has enough columns to
fill the GPU (the full-size layer and training shapes); SDM_WR_CW forces the slice so
that these shapes, which the oracle checks on every stream and token, run the same
kernel: parity with the oracle, chunk-size independence, bitwise repeatability and the
same bits as narrower slices.
"""

import pytest
import torch

import sdm_inputs
from sdm_inputs import CONFIGS
from sdm_testlib import compare_stream, gpu_write_read

pytestmark = pytest.mark.gpu


def _slice_cols(cfg) -> int:
    return 128 // (4 if cfg.bank_dtype == "f32" else 2)


@pytest.fixture
def blocks(monkeypatch):
    def force(cfg):
        monkeypatch.setenv("SDM_WR_CW", str(_slice_cols(cfg)))
    return force


BLOCK_VARIANTS = {
    "tiny": dict(),
    "w64_r64": dict(W=64, R=64, T=40),
    "w48_r64_ragged": dict(W=48, R=64, T=37, chunk_size=5),
    "w128_r96": dict(factor_dims=(64, 64), W=128, R=96, T=40, d_v=32),
    "w3_r5": dict(W=3, R=5, T=30),
    "one_write_one_read": dict(W=1, R=1),
    "bf16_bank": dict(act_dtype="bf16", bank_dtype="bf16", W=64, R=32, T=40),
    "f32_acts_bf16_bank": dict(bank_dtype="bf16", d_v=128, T=32),
    "bf16_acts": dict(act_dtype="bf16", d_v=96, W=24, R=40, T=40),
    "chunk_1": dict(T=40, chunk_size=1, W=32, R=32),
    "every_slot": dict(factor_dims=(4, 4), W=16, R=16, T=24),
    "three_factors": dict(factor_dims=(8, 8, 8), d_sub=16, W=16, R=12),
    "many_streams": dict(B=3, H=2, T=50, W=64, R=64),
    "long_head": dict(d_v=2048, T=24, W=64, R=64),
}


@pytest.mark.parametrize("name", sorted(BLOCK_VARIANTS))
def test_block_layout_matches_oracle(blocks, name):
    kw = dict(BLOCK_VARIANTS[name])
    chunk = kw.pop("chunk_size", None)
    cfg = CONFIGS["tiny"].replace(**kw)
    assert cfg.d_v * (4 if cfg.bank_dtype == "f32" else 2) % 128 == 0
    blocks(cfg)
    d = sdm_inputs.make_inputs(cfg)
    gpu = gpu_write_read(cfg, d, chunk_size=chunk)
    streams = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    res = [compare_stream(cfg, d, gpu, b, h) for (b, h) in streams]
    assert sum(r["near_ties"] for r in res) <= 1


def test_block_layout_chunk_size_changes_nothing(blocks):
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=200)
    blocks(cfg)
    d = sdm_inputs.make_inputs(cfg)
    ref = gpu_write_read(cfg, d, chunk_size=64)
    for c in (1, 3, 17, 128, 256):
        out = gpu_write_read(cfg, d, chunk_size=c)
        for k in ref:
            assert torch.equal(ref[k], out[k]), (c, k)


def test_block_layout_bitwise_repeatable(blocks):
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=120, d_v=256)
    blocks(cfg)
    d = sdm_inputs.make_inputs(cfg)
    first = gpu_write_read(cfg, d)
    for _ in range(2):
        out = gpu_write_read(cfg, d)
        for k in first:
            assert torch.equal(first[k], out[k]), k


def test_results_do_not_depend_on_the_slice_width(monkeypatch):
    # every slice width runs the same block-ordered step: an element's sums depend on
    # W and R only, so 128-byte and 32-byte slices give the same bits
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=60, d_v=128)
    d = sdm_inputs.make_inputs(cfg)
    monkeypatch.setenv("SDM_WR_CW", str(_slice_cols(cfg)))
    wide = gpu_write_read(cfg, d)
    monkeypatch.setenv("SDM_WR_CW", "8")
    narrow = gpu_write_read(cfg, d)
    for k in wide:
        assert torch.equal(wide[k], narrow[k]), k
