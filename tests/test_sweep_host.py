"""Host-side checks of the configuration sweep (no GPU): the candidate list
covers the axes the pages tune (tile shape, pipeline depth, rasterisation
group) plus the split over K, each configuration once, within the limits the
library accepts; shape strings parse as M x N x K or B x M x N x K."""
import itertools

import pytest

import tiled_gemm_tg_gb300 as tg
from tiled_gemm_tg_gb300 import sweep


def test_parse_shapes():
    assert sweep.parse_shapes("1024x2048x512") == [(1024, 2048, 512)]
    assert sweep.parse_shapes("16X4096x4096,256x256x256x256,") == [(16, 4096, 4096),
                                                                  (256, 256, 256, 256)]
    assert sweep.parse_shapes("") == []


@pytest.mark.parametrize("M", [16, 64, 65, 1024])
def test_candidates_cover_every_axis(M):
    cands = sweep.candidates(M, 2048, 512)
    assert len(cands) == len(set(cands)), "a configuration is listed twice"
    pair = [c for c in cands if c[0] == sweep.PAIR]
    main = [c for c in cands if c[0] == sweep.MAIN]
    skinny = [c for c in cands if c[0] == sweep.SKINNY]
    # the pair kernel: groups 2..32 at its default depth, and every shallower depth
    assert {c[2] for c in pair if c[3] == 0} >= {2, 4, 8, 16, 32}
    assert {c[3] for c in pair if c[3] != 0} == set(range(2, sweep.MAX_STAGES[(sweep.PAIR, 0)]))
    for bn in (64, 128, 256):
        mine = [c for c in main if c[1] == bn]
        assert {c[2] for c in mine if c[2] != 0} == {4, 8, 16, 32}
        assert {c[3] for c in mine if c[3] != 0} == set(range(2, sweep.MAX_STAGES[(sweep.MAIN, bn)]))
        assert {c[4] for c in mine} >= {1, 2, 4, 8}
        # a forced group or depth is timed unsplit, so the axes stay separate
        assert all(c[4] == 1 for c in mine if c[2] != 0 or c[3] != 0)
    assert bool(skinny) == (M <= 64)


def test_candidate_values_are_accepted_by_the_library():
    """Every forced value the sweep sends is one the force entry points take
    (the library refuses, with TG_ERR_INVALID_ARG, anything else)."""
    tg.lib()
    try:
        for path, bn, group, stages, split in sweep.candidates(16, 4096, 4096):
            tg.tg_gemm_force_path(path)
            assert tg.tg_gemm_force_tiling(bn, group) == tg.TG_OK
            assert tg.tg_gemm_force_stages(stages) == tg.TG_OK
            assert tg.tg_gemm_force_split_k(split) == tg.TG_OK
    finally:
        tg.tg_gemm_force_path(0)
        tg.tg_gemm_force_tiling(0, 0)
        tg.tg_gemm_force_stages(0)
        tg.tg_gemm_force_split_k(0)


def test_max_stages_match_the_documented_rings():
    """The deepest ring per kernel: the pair kernel 3 stages of 64 KB; the
    one-CTA kernel 4 stages for 256-column tiles (k-block of 64 fp16), 3 for
    128 and 4 for 64 (k-blocks of 128)."""
    assert sweep.MAX_STAGES == {(sweep.PAIR, 0): 3, (sweep.MAIN, 64): 4, (sweep.MAIN, 128): 3,
                                (sweep.MAIN, 256): 4}
    # ring bytes per CTA stay inside 227 KB with the 32 KB epilogue staging
    stage_kb = {64: (16 + 8) * 2, 128: (16 + 16) * 2, 256: 16 + 32}
    for bn, kb in stage_kb.items():
        assert sweep.MAX_STAGES[(sweep.MAIN, bn)] * kb + 32 <= 227
        assert (sweep.MAX_STAGES[(sweep.MAIN, bn)] + 1) * kb + 32 > 227


def test_split_axis_only_on_the_one_cta_kernel():
    for c in itertools.chain(sweep.candidates(16, 4096, 4096), sweep.candidates(4096, 4096, 4096)):
        if c[0] != sweep.MAIN:
            assert c[4] == 0
