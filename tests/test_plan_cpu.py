"""Host logic of the launch planner (nf4_plan_query: no device needed).

The planner is a deterministic function of the shape, the SM count and the
launch options.  These tests pin its decisions on the measured workloads
(GB300: 152 SMs) and check invariants every plan must satisfy: the workspace
it asks for covers what its kernels write, the grid fits the device, stream-K
only where the fused kernel supports it, the launch options take effect.
"""
import itertools

import pytest

from bit_nf4_quantized_linear_gb300 import _lib, build

SMS = 152
FWD, DGRAD = _lib.OP_LINEAR_FWD, _lib.OP_LINEAR_DGRAD


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    _lib.lib()


@pytest.fixture(autouse=True)
def _default_options():
    _lib.set_stream_k(_lib.STREAM_K_AUTO)
    _lib.set_small_m_path(_lib.SMALL_M_AUTO)
    _lib.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)
    yield
    _lib.set_stream_k(_lib.STREAM_K_AUTO)
    _lib.set_small_m_path(_lib.SMALL_M_AUTO)
    _lib.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)


def q(op, M, N, K, sms=SMS, **kw):
    return _lib.plan_query(op, M, N, K, sms, **kw)


def test_plans_of_the_measured_workloads():
    # K = N = 4096 sweep: CTA-pair tiles (512 tokens x 256 rows on two CTAs) from
    # M = 2048, stream-K at 1536, whole 256-token tiles at 1024; at M = 512 a 2-way
    # cluster split (the two halves of a tile on one cluster, no workspace).
    for M, bt, sk in [(1024, 256, 0), (1536, 256, 1), (2048, 512, 0), (4096, 512, 0), (8192, 512, 0)]:
        for op in (FWD, DGRAD):
            p = q(op, M, 4096, 4096)
            assert (p["kernel"], p["token_tile"], p["stream_k"]) == ("fused", bt, sk), (M, p)
    for op in (FWD, DGRAD):
        p = q(op, 512, 4096, 4096)
        assert (p["token_tile"], p["splits"], p["cluster_split"], p["grid"], p["workspace_bytes"]) == \
            (256, 2, 2, 128, 0), p
    # Llama-3.1-8B set at M = 512: k/v forward as 4-way cluster splits of 128-token
    # tiles, k/v input gradient as 2-way cluster splits.
    p = q(FWD, 512, 1024, 4096)
    assert (p["token_tile"], p["cluster_split"]) == (128, 4), p
    p = q(DGRAD, 512, 1024, 4096)
    assert (p["token_tile"], p["cluster_split"], p["stream_k"]) == (256, 2, 0)
    # gate / up forward and down input gradient (224 tiles of 64 steps) on
    # stream-K; their 224-step contractions over 64 tiles (gate / up input
    # gradient, down forward) as 2-way cluster splits.
    for op, N, K in [(FWD, 14336, 4096), (DGRAD, 4096, 14336)]:
        assert q(op, 512, N, K)["stream_k"] == 1
    for op, N, K in [(DGRAD, 14336, 4096), (FWD, 4096, 14336)]:
        p = q(op, 512, N, K)
        assert (p["cluster_split"], p["stream_k"], p["workspace_bytes"]) == (2, 0, 0), p
    # Small M: the warp-MMA kernels for 4-bit codes, bf16 or fp16 operands;
    # one-byte codes always take the fused kernel.
    assert q(FWD, 1, 4096, 4096)["kernel"] == "small_m_mma"
    assert q(DGRAD, 8, 4096, 4096)["kernel"] == "small_m_mma"
    assert q(FWD, 1, 4096, 4096, f16=True)["kernel"] == "small_m_mma"
    assert q(DGRAD, 8, 4096, 4096, f16=True)["kernel"] == "small_m_mma"
    assert q(FWD, 17, 4096, 4096, f16=True)["kernel"] == "fused"
    assert q(FWD, 1, 4096, 4096, bits=8)["kernel"] == "fused"


SHAPES = list(itertools.product([1, 3, 16, 17, 32, 33, 100, 129, 300, 512, 700, 2048, 5000],
                                [64, 320, 1000, 4096], [64, 1024, 4096]))


def test_token_split_of_pair_plans():
    # M = 8192 at K = N = 4096: four rounds of CTA-pair tiles become three (the first
    # 7168 tokens) plus one launch of 256-token tiles over the last 1024; M = 4096
    # and 16384 divide into whole rounds and keep one launch.
    for op in (FWD, DGRAD):
        p = q(op, 8192, 4096, 4096)
        assert (p["token_tile"], p["items"], p["tail_tokens"], p["tail_token_tile"]) == (512, 224, 1024, 256), p
        assert p["workspace_bytes"] == 0
        for M in (2048, 4096, 16384):
            assert q(op, M, 4096, 4096)["tail_tokens"] == 0
    assert q(FWD, 8192, 4096, 4096, bits=8)["tail_tokens"] == 0   # (no pairs for one-byte codes)
    # the parts of a split run whole contractions: no workspace, whatever the shape
    # (the 32B-shaped stack splits several of its products at M = 4096)
    seen = 0
    for M in (2048, 4096, 6144, 8192, 12288):
        for N, K in ((5120, 5120), (1024, 5120), (27648, 5120), (5120, 27648), (14336, 4096), (4096, 14336)):
            for op in (FWD, DGRAD):
                p = q(op, M, N, K)
                if p["tail_tokens"]:
                    seen += 1
                    assert p["workspace_bytes"] == 0 and p["tail_token_tile"] == 256, (M, N, K, op, p)
                    assert p["tail_tokens"] % 512 == 0 and p["tail_tokens"] < M
    assert seen > 0
    _lib.set_token_tile(512)
    try:
        assert q(FWD, 8192, 4096, 4096)["tail_tokens"] == 0        # a fixed tile is never split
    finally:
        _lib.set_token_tile(0)


@pytest.mark.parametrize("bits,f16", [(4, False), (8, False), (4, True)])
def test_plan_invariants(bits, f16):
    for (M, N, K), op in itertools.product(SHAPES, (FWD, DGRAD)):
        p = q(op, M, N, K, bits=bits, f16=f16)
        assert p == q(op, M, N, K, bits=bits, f16=f16)  # deterministic
        ncols, contract = (N, K) if op == FWD else (K, N)
        if bits == 8:
            assert p["kernel"] == "fused"
        if f16:  # fp16: the warp-MMA kernels or the fused kernel, never the SIMT GEMV
            assert p["kernel"] in ("fused", "small_m_mma")
        if p["kernel"] != "fused":
            assert M <= 16 and p["workspace_bytes"] >= 0
            continue
        bt = p["token_tile"]
        assert bt in (16, 32, 64, 128, 256, 512) and (bits == 4 or bt <= 128)
        assert 1 <= p["grid"] <= SMS
        ttiles = -(-(M - p["tail_tokens"]) // bt)
        wtiles = -(-ncols // (256 if bt == 512 else 128))  # CTA pairs: 256-row weight tiles
        if bt == 512:
            assert M >= 1024 and p["grid"] % 2 == 0 and not p["stream_k"] and not p["cluster_split"]
        assert p["items"] == wtiles * ttiles * p["splits"]
        assert p["splits"] <= max(1, -(-contract // 64))
        if p["cluster_split"]:
            cs = p["cluster_split"]
            # one tile per cluster of cs CTAs, in one wave, no workspace
            assert cs in (2, 4, 8) and p["splits"] == cs and bits == 4 and bt // cs >= 32
            assert p["grid"] == p["items"] and p["grid"] % cs == 0 and p["workspace_bytes"] == 0
            assert not p["stream_k"]
        elif p["stream_k"]:
            assert p["splits"] == 1
            # one partial tile [4 row quarters][bt tokens][32 rows] fp32 per CTA, then
            # one 8-byte ready flag per CTA and row quarter
            assert p["workspace_bytes"] == p["grid"] * 128 * bt * 4 + p["grid"] * 4 * 8
            assert p["grid"] == min(SMS, p["items"] * -(-contract // 64))
        elif p["splits"] > 1:
            assert p["workspace_bytes"] == p["splits"] * M * ncols * 4
        else:
            assert p["workspace_bytes"] == 0


def test_launch_options_take_effect():
    _lib.set_stream_k(_lib.STREAM_K_OFF)
    assert all(q(op, M, 4096, 4096)["stream_k"] == 0
               for op in (FWD, DGRAD) for M in (512, 1536, 2048, 4096))
    _lib.set_stream_k(_lib.STREAM_K_FORCE)
    for M in (33, 129, 700, 8192):
        p = q(FWD, M, 1000, 1024)
        assert p["stream_k"] == 1 and p["splits"] == 1, (M, p)
    _lib.set_stream_k(_lib.STREAM_K_AUTO)
    _lib.set_small_m_path(_lib.SMALL_M_SIMT)
    assert q(FWD, 4, 4096, 4096)["kernel"] == "simt_gemv"
    _lib.set_small_m_path(_lib.SMALL_M_TILES)
    assert q(FWD, 4, 4096, 4096)["kernel"] == "fused"
    _lib.set_small_m_path(_lib.SMALL_M_AUTO)
    _lib.set_cluster_split(_lib.CLUSTER_SPLIT_OFF)
    assert all(q(op, M, N, 4096)["cluster_split"] == 0
               for op in (FWD, DGRAD) for M in (128, 512) for N in (1024, 4096))
    _lib.set_cluster_split(_lib.CLUSTER_SPLIT_FORCE)
    for M, N, K in [(64, 4096, 4096), (300, 200, 256), (512, 14336, 4096)]:
        p = q(FWD, M, N, K)
        tiles = -(-N // 128) * -(-M // p["token_tile"])
        assert p["cluster_split"] > 1 or tiles * 2 > SMS, (M, N, K, p)
    _lib.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)


def test_fixed_token_tile_option():
    # A fixed tile is the only candidate for M > 32 (one-byte codes: at most 128),
    # on every schedule; other values are ignored; 0 restores the planner's choice.
    try:
        for bt in (64, 128, 256, 512):
            _lib.set_token_tile(bt)
            tw = 256 if bt == 512 else 128
            for M, N, K in [(33, 256, 512), (700, 640, 1024), (4096, 4096, 4096)]:
                for op in (FWD, DGRAD):
                    p = q(op, M, N, K)
                    assert p["token_tile"] == bt, (bt, M, p)
                    assert p["items"] == -(-(N if op == FWD else K) // tw) * -(-M // bt) * p["splits"]
            assert q(FWD, 700, 640, 1024, bits=8)["token_tile"] == min(bt, 128)
            assert q(FWD, 20, 640, 1024)["token_tile"] == 32  # M <= 32 keeps its own tile
        _lib.set_stream_k(_lib.STREAM_K_FORCE)
        _lib.set_token_tile(128)
        p = q(FWD, 4096, 4096, 4096)
        assert p["stream_k"] and p["token_tile"] == 128
        _lib.set_stream_k(_lib.STREAM_K_AUTO)
        _lib.set_token_tile(96)  # ignored
        assert q(FWD, 4096, 4096, 4096)["token_tile"] == 128
        _lib.set_token_tile(512)  # CTA-pair tiles: 256-row weight tiles, two CTAs per item
        p = q(FWD, 700, 640, 1024)
        assert p["token_tile"] == 512 and p["items"] == 3 * 2 * p["splits"] and not p["stream_k"]
        assert p["grid"] % 2 == 0 and p["grid"] <= SMS
        assert q(FWD, 700, 640, 1024, bits=8)["token_tile"] == 128
    finally:
        _lib.set_token_tile(0)
        _lib.set_stream_k(_lib.STREAM_K_AUTO)
    assert q(FWD, 4096, 4096, 4096)["token_tile"] == 512


def test_sm_count_changes_the_schedule_not_the_contract():
    # Fewer SMs: more waves; the plan stays within the device and keeps its
    # workspace rules (checked above); it never needs a GPU to compute.
    for sms in (1, 8, 76, 148, 152, 160):
        for M in (64, 2048):
            p = q(FWD, M, 4096, 4096, sms=sms)
            assert 1 <= p["grid"] <= sms


@pytest.mark.parametrize("args", [
    (0, 8, 64, 64, SMS, 4, 0),            # not a dense product
    (FWD, 0, 64, 64, SMS, 4, 0),          # empty M
    (FWD, 8, 64, 64, 0, 4, 0),            # no SMs
    (FWD, 8, 64, 64, SMS, 6, 0),          # code width
    (FWD, 8, 64, 64, SMS, 8, 1),          # fp16 with one-byte codes
])
def test_plan_query_rejects_bad_arguments(args):
    op, M, N, K, sms, bits, f16 = args
    with pytest.raises(_lib.NF4Error):
        _lib.plan_query(op, M, N, K, sms, bits=bits, f16=bool(f16))
