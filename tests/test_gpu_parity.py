"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Bit-exact: packed codes, absmax, nested statistics, dense dequantisation, and the
identity probe (a one-hot activation selects one dequantised weight exactly).
Within tolerance (relative Frobenius <= 5e-3, per element <= 1e-2 (|ref| + rms)):
the forward and input-gradient products against the oracle's fp64 sums.
Bit-identical across reruns.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import codebooks as ocb
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import _lib, ops
from bit_nf4_quantized_linear_gb300 import synth
from tests.helpers import bf16_bits, oracle_state, parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    nf4.device_check()
    nf4.device_status(clear=True)
    yield
    assert nf4.device_status() == 0, "a kernel recorded a device error"


def _quant_pair(N, K, dq, seed=0, code8=None, dtype=torch.float32):
    g = synth.generator(seed)
    w32 = synth.weight(N, K, g)
    if dtype == torch.bfloat16:
        w32 = w32.to(torch.bfloat16).float()
    w = nf4.quantize(w32.to(DEV, dtype), double_quant=dq,
                     code8=None if code8 is None else torch.from_numpy(code8))
    st = oracle_state(w32, dq, code8)
    return w, st, g


def _assert_state_equal(w, st):
    np.testing.assert_array_equal(w.packed.cpu().numpy(), st.packed)
    np.testing.assert_array_equal(w.absmax.cpu().numpy().view(np.uint32), st.absmax.view(np.uint32))
    if st.double_quant:
        np.testing.assert_array_equal(w.absmax_q.cpu().numpy(), st.absmax_q)
        np.testing.assert_array_equal(w.nested_absmax.cpu().numpy().view(np.uint32),
                                      st.nested_absmax.view(np.uint32))
        np.testing.assert_array_equal(w.nested_offset.cpu().numpy().view(np.uint32),
                                      st.nested_offset.view(np.uint32))


# ------------------------------------------------------- quantise / dequantise --

@pytest.mark.parametrize("N,K,dq", [(64, 64, False), (256, 512, True), (1024, 1024, False),
                                    (4096, 4096, True), (3, 100, True), (1, 17, False),
                                    (1000, 1344, True)])
def test_quantize_bit_exact(N, K, dq):
    w, st, _ = _quant_pair(N, K, dq)
    torch.cuda.synchronize()
    _assert_state_equal(w, st)


def test_quantize_bf16_input_and_linear_code8():
    w, st, _ = _quant_pair(512, 768, True, code8=ocb.linear_code8(), dtype=torch.bfloat16)
    _assert_state_equal(w, st)


@pytest.mark.parametrize("N,K,dq", [(256, 512, True), (1024, 1024, False), (5, 77, True)])
def test_dequantize_bit_exact(N, K, dq):
    w, st, _ = _quant_pair(N, K, dq)
    f32 = nf4.dequantize(w, torch.float32).cpu().numpy().reshape(-1)
    b16 = bf16_bits(nf4.dequantize(w, torch.bfloat16)).reshape(-1)
    np.testing.assert_array_equal(f32.view(np.uint32), oracle.dequantize(st, "f32").reshape(-1).view(np.uint32))
    np.testing.assert_array_equal(b16, oracle.dequantize(st, "bf16").reshape(-1))


# ------------------------------------------------------------------ products --

SMALL = [  # (M, N, K): several tiles, ragged tails, every token-tile width
    (1, 256, 256), (5, 384, 512), (16, 128, 1024), (17, 200, 192), (40, 320, 192),
    (64, 640, 256), (100, 1000, 640), (128, 256, 128), (129, 384, 320), (300, 200, 256),
    (700, 640, 1024),
]


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("dq", [False, True])
def test_fwd_dgrad_parity_small(M, N, K, dq):
    w, st, g = _quant_pair(N, K, dq, seed=M + N + K)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("K,N", [(128, 256), (256, 384), (1024, 512)])
def test_identity_probe_fwd_exact(K, N):
    # x = I_K: y[m, n] = Wb[n, m] exactly, so the in-kernel dequantisation is
    # checked bit for bit (large token tiles), and again with 16 one-hot rows
    # (the split-contraction path).
    w, st, _ = _quant_pair(N, K, True, seed=K)
    wb = oracle.dequantize(st, "bf16")
    eye = torch.eye(K, dtype=torch.bfloat16)
    y = nf4.linear_fwd(eye.to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(y), np.ascontiguousarray(wb.T))
    y16 = nf4.linear_fwd(eye[:16].contiguous().to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(y16), np.ascontiguousarray(wb.T[:16]))


@pytest.mark.parametrize("N,K", [(128, 256), (384, 256), (1024, 512)])
def test_identity_probe_dgrad_exact(N, K):
    w, st, _ = _quant_pair(N, K, True, seed=N)
    wb = oracle.dequantize(st, "bf16")
    eye = torch.eye(N, dtype=torch.bfloat16)
    gx = nf4.linear_dgrad(eye.to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(gx), wb)
    gx16 = nf4.linear_dgrad(eye[:16].contiguous().to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(gx16), wb[:16])


@pytest.mark.parametrize("M", [1, 40, 700])
def test_reruns_bit_identical(M):
    N, K = 1024, 1024
    w, st, g = _quant_pair(N, K, True, seed=3)
    x = synth.activation(M, K, g).to(DEV)
    gy = synth.activation(M, N, g).to(DEV)
    y0, gx0 = nf4.linear_fwd(x, w), nf4.linear_dgrad(gy, w)
    for _ in range(10):
        assert torch.equal(nf4.linear_fwd(x, w).view(torch.int16), y0.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy, w).view(torch.int16), gx0.view(torch.int16))


def test_strided_activation_and_output():
    N, K, M = 256, 320, 33
    w, st, g = _quant_pair(N, K, False, seed=5)
    xbig = synth.activation(M, K + 64, g)
    x = xbig[:, 32:32 + K]
    ybig = torch.zeros(M, N + 8, dtype=torch.bfloat16, device=DEV)
    nf4.linear_fwd(xbig.to(DEV)[:, 32:32 + K], w, out=ybig[:, :N])
    parity(ybig[:, :N], oracle.linear_fwd(bf16_bits(x.contiguous()), oracle.dequantize(st, "bf16")))
    assert torch.all(ybig[:, N:] == 0)


def test_empty_batch_is_noop():
    w, _, _ = _quant_pair(128, 128, True)
    y = nf4.linear_fwd(torch.empty(0, 128, dtype=torch.bfloat16, device=DEV), w)
    assert y.shape == (0, 128)


def test_errors_are_reported():
    w, _, _ = _quant_pair(128, 128, False)
    x = torch.zeros(4, 129, dtype=torch.bfloat16, device=DEV)[:, 1:]  # 2-byte offset
    with pytest.raises(nf4.ops._lib.NF4Error) as e:
        nf4.linear_fwd(x, w)
    assert e.value.code == 3
    with pytest.raises(ValueError):
        nf4.linear_fwd(torch.zeros(4, 128, dtype=torch.bfloat16), w)  # CPU tensor: no CPU path


# ----------------------------------------------------------- full-size sampled --

def _sampled_rows(M, n=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows |= {0, M - 1}
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("M", synth.M_SWEEP)
def test_m_sweep_4096_sampled(M):
    N = K = 4096
    w, st, g = _quant_pair(N, K, True, seed=11)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    rows = _sampled_rows(M)
    parity(y[torch.from_numpy(rows).to(DEV)], oracle.linear_fwd(bf16_bits(x), wb, rows), f"fwd M={M}")
    parity(gx[torch.from_numpy(rows).to(DEV)], oracle.linear_dgrad(bf16_bits(gy), wb, rows), f"dgrad M={M}")


@pytest.mark.parametrize("name,K,N", synth.LLAMA8B_PROJ)
def test_llama8b_projection_set_sampled(name, K, N):
    M = 512
    w, st, g = _quant_pair(N, K, True, seed=hash(name) % 1000)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    rows = _sampled_rows(M, 4)
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    parity(y[torch.from_numpy(rows).to(DEV)], oracle.linear_fwd(bf16_bits(x), wb, rows), name)
    parity(gx[torch.from_numpy(rows).to(DEV)], oracle.linear_dgrad(bf16_bits(gy), wb, rows), name)


def test_config1_single_linear_full():
    # x [256, 1024], W [1024, 1024], fp32 absmax: compared in full.
    w, st, g = _quant_pair(1024, 1024, False, seed=0)
    x = synth.activation(256, 1024, g)
    gy = synth.activation(256, 1024, g)
    wb = oracle.dequantize(st, "bf16")
    parity(nf4.linear_fwd(x.to(DEV), w), oracle.linear_fwd(bf16_bits(x), wb), "cfg1 fwd")
    parity(nf4.linear_dgrad(gy.to(DEV), w), oracle.linear_dgrad(bf16_bits(gy), wb), "cfg1 dgrad")


# ------------------------------------------------------------------- grouped --

def _grouped_case(E, N_e, K, tokens, topk, dq, seed):
    g = synth.generator(seed)
    w32 = synth.weight(E * N_e, K, g)
    row_token, offsets = synth.routing(tokens, E, topk, g)
    xt = synth.activation(tokens, K, g)
    x = xt[row_token].contiguous()
    T = x.shape[0]
    gy = synth.activation(T, N_e, g)
    w = nf4.quantize(w32.to(DEV), double_quant=dq)
    st = oracle_state(w32, dq)
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    return w, wb, x, gy, offsets


@pytest.mark.parametrize("dq", [False, True])
def test_grouped_small_ragged(dq):
    E, N_e, K = 6, 192, 256
    w, wb, x, gy, offsets = _grouped_case(E, N_e, K, 50, 2, dq, seed=21)
    offs = offsets.numpy()
    y = nf4.grouped_fwd(x.to(DEV), offsets.to(DEV), w, E)
    gx = nf4.grouped_dgrad(gy.to(DEV), offsets.to(DEV), w, E)
    parity(y, oracle.grouped_fwd(bf16_bits(x), offs, wb), "grouped fwd")
    parity(gx, oracle.grouped_dgrad(bf16_bits(gy), offs, wb), "grouped dgrad")


@pytest.mark.parametrize("proj", ["gate", "down"])
def test_grouped_olmoe_experts(proj):
    c = synth.OLMOE
    E = c["experts"]
    N_e, K = (c["inter"], c["hidden"]) if proj == "gate" else (c["hidden"], c["inter"])
    w, wb, x, gy, offsets = _grouped_case(E, N_e, K, c["tokens"], c["topk"], False, seed=31)
    offs = offsets.numpy()
    y = nf4.grouped_fwd(x.to(DEV), offsets.to(DEV), w, E)
    gx = nf4.grouped_dgrad(gy.to(DEV), offsets.to(DEV), w, E)
    parity(y, oracle.grouped_fwd(bf16_bits(x), offs, wb), f"olmoe {proj} fwd")
    parity(gx, oracle.grouped_dgrad(bf16_bits(gy), offs, wb), f"olmoe {proj} dgrad")


def test_grouped_empty_experts_and_bad_offsets():
    E, N_e, K = 4, 128, 128
    w, wb, x, gy, _ = _grouped_case(E, N_e, K, 20, 1, False, seed=41)
    offs = np.array([0, 0, 20, 20, 20], dtype=np.int32)
    y = nf4.grouped_fwd(x.to(DEV), torch.from_numpy(offs).to(DEV), w, E)
    parity(y, oracle.grouped_fwd(bf16_bits(x), offs, wb), "empty experts")
    nf4.device_status(clear=True)
    bad = torch.tensor([0, 15, 5, 20, 20], dtype=torch.int32, device=DEV)
    nf4.grouped_fwd(x.to(DEV), bad, w, E)
    torch.cuda.synchronize()
    assert nf4.device_status(clear=True) == 8


# ------------------------------------------------------------------ small M --
# M <= 16: the tensor-core small-M kernels by default (warp-level MMA over a
# shared dequantisation table, contraction split over thread-block clusters);
# the SIMT GEMV and the split tcgen05 tiles on request.

SMALL_M = [(1, 64, 64), (2, 104, 128), (3, 136, 1088), (4, 4096, 1024), (5, 296, 2112),
           (7, 200, 2112), (8, 96, 5120), (1, 4096, 14336), (2, 14336, 4096), (6, 4096, 14336),
           (9, 520, 2112), (13, 1000, 4096), (16, 4096, 4096)]


@pytest.fixture
def restore_small_m():
    yield
    ops.set_small_m_path(_lib.SMALL_M_AUTO)
    ops.set_weight_prefetch(False)


@pytest.mark.parametrize("M,N,K", SMALL_M)
@pytest.mark.parametrize("dq", [False, True])
def test_small_m_default_path_parity(M, N, K, dq):
    w, st, g = _quant_pair(N, K, dq, seed=7 * M + N + K)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    c = nf4.path_counters()
    if M <= 8:
        assert c["skinny_fwd"] == 1 and c["skinny_dgrad"] == 1, c
    assert c["skinny_fwd"] + c["gemv_fwd"] + c["linear_fwd"] == 1
    assert c["skinny_dgrad"] + c["gemv_dgrad"] + c["linear_dgrad"] == 1
    parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"small-M fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"small-M dgrad {M}x{N}x{K}")
    assert torch.equal(nf4.linear_fwd(x.to(DEV), w).view(torch.int16), y.view(torch.int16))
    assert torch.equal(nf4.linear_dgrad(gy.to(DEV), w).view(torch.int16), gx.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (3, 136, 1088), (4, 4096, 1024), (2, 14336, 4096),
                                   (12, 296, 2112)])
def test_small_m_simt_and_tile_paths(M, N, K, restore_small_m):
    w, st, g = _quant_pair(N, K, True, seed=3 * M + N + K)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    for path in (_lib.SMALL_M_SIMT, _lib.SMALL_M_TILES):
        ops.set_small_m_path(path)
        nf4.reset_path_counters()
        y = nf4.linear_fwd(x.to(DEV), w)
        gx = nf4.linear_dgrad(gy.to(DEV), w)
        c = nf4.path_counters()
        assert c["skinny_fwd"] == 0 and c["skinny_dgrad"] == 0
        if path == _lib.SMALL_M_SIMT and M <= 4:
            assert c["gemv_fwd"] == 1 and c["gemv_dgrad"] == 1
        else:
            assert c["linear_fwd"] == 1 and c["linear_dgrad"] == 1
        parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"path {path} fwd {M}x{N}x{K}")
        parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"path {path} dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("N,K", [(64, 128), (296, 2048), (4096, 4096)])
@pytest.mark.parametrize("path", [0, 1])
def test_small_m_identity_probe_exact(N, K, path, restore_small_m):
    """One-hot activations read single weight values back: the small-M operands
    are exactly the dequantised bf16 weights."""
    ops.set_small_m_path(path)
    w, st, _ = _quant_pair(N, K, True, seed=N + K)
    wb = oracle.dequantize(st, "bf16")
    eye = torch.eye(K, dtype=torch.bfloat16)[:4].contiguous()
    y = nf4.linear_fwd(eye.to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(y), np.ascontiguousarray(wb.T[:4]))
    eyen = torch.eye(N, dtype=torch.bfloat16)[:4].contiguous()
    gx = nf4.linear_dgrad(eyen.to(DEV), w)
    np.testing.assert_array_equal(bf16_bits(gx), wb[:4])


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (8, 4096, 14336), (16, 1024, 4096),
                                   (64, 4096, 4096), (512, 1024, 4096), (1536, 4096, 4096)])
def test_weight_prefetch_leaves_results_unchanged(M, N, K, restore_small_m):
    """Reading the frozen weight before the grid dependency resolves changes only
    timing: outputs are bit-identical with and without it, also back to back
    (small-M kernels; the fused kernel with a contraction split, classic and
    stream-K schedules)."""
    g = synth.generator(M + K)
    w = nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=True)
    x = synth.activation(M, K, g).to(DEV)
    gy = synth.activation(M, N, g).to(DEV)
    outs = []
    for pf in (False, True):
        ops.set_weight_prefetch(pf)
        y1 = nf4.linear_fwd(x, w)
        g1 = nf4.linear_dgrad(gy, w)
        y2 = nf4.linear_fwd(x, w)   # starts while the previous kernel drains
        outs.append((y1, g1, y2))
    for t in range(3):
        assert torch.equal(outs[0][t].view(torch.int16), outs[1][t].view(torch.int16))
    assert torch.equal(outs[0][0].view(torch.int16), outs[0][2].view(torch.int16))


@pytest.mark.parametrize("M,N,K,mode", [(512, 4096, 4096, 0), (512, 4096, 4096, 1), (1024, 640, 1024, 0),
                                        (700, 384, 2048, 1), (2048, 14336, 4096, 0)])
def test_wide_tiles_classic_and_stream_k_match_oracle(M, N, K, mode, restore_stream_k):
    # 256-token tiles on both schedules of the fused kernel: sampled rows against
    # the oracle, each schedule bit-identical on a rerun.
    w, st, g = _quant_pair(N, K, True, seed=M + N)
    a = synth.activation(M, K if mode == 0 else N, g)
    wb = oracle.dequantize(st, "bf16")
    rows = _sampled_rows(M, 5)
    ref = (oracle.linear_fwd if mode == 0 else oracle.linear_dgrad)(bf16_bits(a), wb, rows)
    f = nf4.linear_fwd if mode == 0 else nf4.linear_dgrad
    for sk in (_lib.STREAM_K_OFF, _lib.STREAM_K_FORCE):
        ops.set_stream_k(sk)
        o = f(a.to(DEV), w)
        parity(o[torch.from_numpy(rows).to(DEV)], ref, f"stream_k={sk} mode={mode} M={M}")
        assert torch.equal(f(a.to(DEV), w).view(torch.int16), o.view(torch.int16))


# --------------------------------------------------------------- fp4 codebook --
# The "fp4" quant_type runs the same kernels with the E2M1 levels as code4.

def _quant_pair_fp4(N, K, dq, seed=0):
    g = synth.generator(seed)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=dq, quant_type="fp4")
    st = oracle.quantize(w32.numpy(), ocb.fp4_code4(), 64, dq, ocb.dynamic_code8(), 256)
    return w, st, g


@pytest.mark.parametrize("N,K,dq", [(256, 512, True), (1000, 1344, False), (4096, 4096, True)])
def test_fp4_quantize_dequantize_bit_exact(N, K, dq):
    w, st, _ = _quant_pair_fp4(N, K, dq, seed=N)
    torch.cuda.synchronize()
    _assert_state_equal(w, st)
    f32 = nf4.dequantize(w, torch.float32).cpu().numpy().reshape(-1)
    b16 = bf16_bits(nf4.dequantize(w, torch.bfloat16)).reshape(-1)
    np.testing.assert_array_equal(f32.view(np.uint32), oracle.dequantize(st, "f32").reshape(-1).view(np.uint32))
    np.testing.assert_array_equal(b16, oracle.dequantize(st, "bf16").reshape(-1))


@pytest.mark.parametrize("M", [1, 8, 40, 300])
def test_fp4_fwd_dgrad_parity(M):
    N, K = 640, 1024
    w, st, g = _quant_pair_fp4(N, K, True, seed=M)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    parity(nf4.linear_fwd(x.to(DEV), w), oracle.linear_fwd(bf16_bits(x), wb), f"fp4 fwd M={M}")
    parity(nf4.linear_dgrad(gy.to(DEV), w), oracle.linear_dgrad(bf16_bits(gy), wb), f"fp4 dgrad M={M}")


def test_fp4_identity_probe_exact():
    # One-hot rows select single dequantised weights; values compare exactly (a
    # -0 weight sums to +0 with the other products, so values, not bits).
    K, N = 256, 384
    w, st, _ = _quant_pair_fp4(N, K, True, seed=5)
    wb = oracle.dequantize(st, "bf16")
    wbf = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).float().numpy()
    for rows in (K, 16):
        eye = torch.eye(K, dtype=torch.bfloat16)[:rows].contiguous()
        y = nf4.linear_fwd(eye.to(DEV), w).float().cpu().numpy()
        np.testing.assert_array_equal(y, np.ascontiguousarray(wbf.T[:rows]))


# ------------------------------------------------------------------- stream-K --
# Forced on small shapes, tiles are cut between many CTAs (a tile's first segment
# adds up to several following partials), which exercises every case of the
# schedule; the default planner picks it for the large-M sweep points above.

@pytest.fixture
def restore_stream_k():
    yield
    ops.set_stream_k(_lib.STREAM_K_AUTO)


@pytest.mark.parametrize("M,N,K", [(40, 320, 192), (64, 1000, 640), (129, 384, 320),
                                   (300, 640, 1024), (700, 640, 1024)])
def test_stream_k_forced_parity_and_reruns(M, N, K, restore_stream_k):
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    w, st, g = _quant_pair(N, K, True, seed=7 * M + N)
    x = synth.activation(M, K, g).to(DEV)
    gy = synth.activation(M, N, g).to(DEV)
    wb = oracle.dequantize(st, "bf16")
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x, w)
    gx = nf4.linear_dgrad(gy, w)
    c = nf4.path_counters()
    assert c["stream_k"] == 2 and c["splitk_reduce"] == 0, c
    parity(y, oracle.linear_fwd(bf16_bits(x.cpu()), wb), f"stream-K fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy.cpu()), wb), f"stream-K dgrad {M}x{N}x{K}")
    for _ in range(5):
        assert torch.equal(nf4.linear_fwd(x, w).view(torch.int16), y.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy, w).view(torch.int16), gx.view(torch.int16))


def test_stream_k_wait_that_runs_out_reports_timeout(restore_stream_k):
    """Failure detection without a fault: the injected launch's finishing CTAs wait
    for a flag value no CTA publishes; the bounded waits (2 s) run out, the kernel
    records NF4_ERR_TIMEOUT and exits, and the next launch is normal and correct."""
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    M, N, K = 300, 640, 1024
    w, st, g = _quant_pair(N, K, True, seed=5)
    x = synth.activation(M, K, g).to(DEV)
    nf4.device_status(clear=True)
    nf4.reset_path_counters()
    ops.inject_stream_k_timeout()
    nf4.linear_fwd(x, w)
    torch.cuda.synchronize()
    assert nf4.path_counters()["stream_k"] == 1
    assert nf4.device_status(clear=True) == 6  # NF4_ERR_TIMEOUT
    y = nf4.linear_fwd(x, w)
    torch.cuda.synchronize()
    assert nf4.device_status() == 0
    parity(y, oracle.linear_fwd(bf16_bits(x.cpu()), oracle.dequantize(st, "bf16")),
           "stream-K launch after a timed-out one")


def test_stream_k_concurrent_products_on_two_streams(restore_stream_k):
    """Two stream-K products at once on two streams, each with its own workspace:
    one launch's CTAs can find SMs held by the other's.  A CTA waits only for CTAs
    of lower index of its own launch, so both finish without a timeout, match the
    oracle and repeat bit for bit."""
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    M, N, K = 2048, 4096, 4096
    w1, st1, g1 = _quant_pair(N, K, True, seed=61)
    w2, st2, g2 = _quant_pair(N, K, True, seed=62)
    x1 = synth.activation(M, K, g1)
    gy2 = synth.activation(M, N, g2)
    x1d, gy2d = x1.to(DEV), gy2.to(DEV)
    nf4.device_status(clear=True)
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    ys, gxs = [], []
    for _ in range(4):
        with torch.cuda.stream(s1):
            ys.append(nf4.linear_fwd(x1d, w1))
        with torch.cuda.stream(s2):
            gxs.append(nf4.linear_dgrad(gy2d, w2))
    torch.cuda.synchronize()
    assert nf4.device_status() == 0
    rows = _sampled_rows(M, 5)
    r = torch.from_numpy(rows).to(DEV)
    parity(ys[0][r], oracle.linear_fwd(bf16_bits(x1), oracle.dequantize(st1, "bf16"), rows), "concurrent fwd")
    parity(gxs[0][r], oracle.linear_dgrad(bf16_bits(gy2), oracle.dequantize(st2, "bf16"), rows),
           "concurrent dgrad")
    for i in range(1, 4):
        assert torch.equal(ys[i].view(torch.int16), ys[0].view(torch.int16))
        assert torch.equal(gxs[i].view(torch.int16), gxs[0].view(torch.int16))


def test_stream_k_graph_replays_between_eager_launches(restore_stream_k):
    """A stream-K product captured in a CUDA graph keeps its launch epoch on every
    replay; its ready flags sit in the graph's own workspace and are cleared by the
    CTAs that finish the tiles, so replays interleaved with eager launches of the
    same shape (other workspaces, new epochs) all give the same bits."""
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    M, N, K = 700, 1024, 2048
    w, st, g = _quant_pair(N, K, True, seed=63)
    x = synth.activation(M, K, g).to(DEV)
    ref = nf4.linear_fwd(x, w)
    y = torch.empty_like(ref)
    ws = torch.empty(max(ops.workspace_size(_lib.OP_LINEAR_FWD, M, N, K), 16), dtype=torch.uint8,
                     device=DEV)
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.linear_fwd(x, w, out=y, ws=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ops.linear_fwd(x, w, out=y, ws=ws)
    nf4.device_status(clear=True)
    for _ in range(4):
        y.zero_()
        graph.replay()
        eager = nf4.linear_fwd(x, w)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(eager.view(torch.int16), ref.view(torch.int16))
    assert nf4.device_status() == 0
    parity(ref, oracle.linear_fwd(bf16_bits(x.cpu()), oracle.dequantize(st, "bf16")), "graph stream-K")


@pytest.fixture
def restore_cluster_split():
    yield
    ops.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)


@pytest.mark.parametrize("M,N,K", [(512, 4096, 4096), (512, 1024, 4096), (129, 384, 320), (64, 4096, 1024),
                                   (700, 640, 1024), (300, 200, 256), (256, 2048, 2048)])
def test_cluster_split_parity_and_reruns(M, N, K, restore_cluster_split):
    """Cluster split forced: the contraction slices of a tile run on the CTAs of one
    cluster and the owners add the partials they receive through distributed shared
    memory in rank order.  Both products against the oracle, bit-identical reruns."""
    ops.set_cluster_split(_lib.CLUSTER_SPLIT_FORCE)
    w, st, g = _quant_pair(N, K, True, seed=5 * M + N + K)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    sms = nf4.device_check()
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    c = nf4.path_counters()
    expect = sum(ops.plan_query(op, M, N, K, sms)["cluster_split"] > 1
                 for op in (_lib.OP_LINEAR_FWD, _lib.OP_LINEAR_DGRAD))
    assert expect >= 1 and c["cluster_split"] == expect and c["splitk_reduce"] == 0, c
    parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"cluster split fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"cluster split dgrad {M}x{N}x{K}")
    for _ in range(3):
        assert torch.equal(nf4.linear_fwd(x.to(DEV), w).view(torch.int16), y.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy.to(DEV), w).view(torch.int16), gx.view(torch.int16))
    assert nf4.device_status() == 0


def test_cluster_split_fp16_and_identity_probe(restore_cluster_split):
    ops.set_cluster_split(_lib.CLUSTER_SPLIT_FORCE)
    N, K = 384, 256
    w, st, g = _quant_pair(N, K, True, seed=71)
    wb = oracle.dequantize(st, "bf16")
    nf4.reset_path_counters()
    y = nf4.linear_fwd(torch.eye(K, dtype=torch.bfloat16, device=DEV), w)
    gx = nf4.linear_dgrad(torch.eye(N, dtype=torch.bfloat16, device=DEV), w)
    assert nf4.path_counters()["cluster_split"] == 2
    np.testing.assert_array_equal(bf16_bits(y), np.ascontiguousarray(wb.T))
    np.testing.assert_array_equal(bf16_bits(gx), wb)
    M = 200
    x = synth.activation(M, K, g).float().half()
    yh = nf4.linear_fwd(x.to(DEV), w)
    parity(yh, oracle.linear_fwd(_f16_bits(x), oracle.dequantize_f16(st), dtype="f16"), "cluster split f16")


def test_cluster_split_off_and_on_agree_within_tolerance(restore_cluster_split):
    M, N, K = 512, 4096, 4096
    w, st, g = _quant_pair(N, K, True, seed=72)
    x = synth.activation(M, K, g).to(DEV)
    ys = []
    for mode in (_lib.CLUSTER_SPLIT_OFF, _lib.CLUSTER_SPLIT_FORCE):
        ops.set_cluster_split(mode)
        ys.append(nf4.linear_fwd(x, w).float())
    rel = (torch.linalg.norm(ys[0] - ys[1]) / torch.linalg.norm(ys[0])).item()
    assert rel < 1e-3, rel


def test_stream_k_off_and_on_agree_within_tolerance(restore_stream_k):
    M, N, K = 1536, 1024, 1024
    w, st, g = _quant_pair(N, K, True, seed=11)
    x = synth.activation(M, K, g).to(DEV)
    ys = []
    for mode in (_lib.STREAM_K_OFF, _lib.STREAM_K_FORCE):
        ops.set_stream_k(mode)
        ys.append(nf4.linear_fwd(x, w).float())
    # Only the fp32 summation order differs (the split tiles add partials), so the
    # bf16 results agree except where that order flips a rounding: one bf16 ulp,
    # plus the fp32 sums' own difference (about sqrt(K) 2^-24 of the terms, far
    # below 1e-4 rms) where cancellation leaves a small result.
    rel = (torch.linalg.norm(ys[0] - ys[1]) / torch.linalg.norm(ys[0])).item()
    assert rel < 1e-3, rel
    assert (ys[0] == ys[1]).float().mean().item() > 0.9
    rms = ys[0].pow(2).mean().sqrt()
    bound = torch.maximum(ys[0].abs(), ys[1].abs()) * 2.0 ** -7 + 1e-4 * rms
    assert bool(((ys[0] - ys[1]).abs() <= bound).all())


# ------------------------------------------------------- 8-bit weight storage --
# "int8" (blockwise dynamic map) and "fp8" (e4m3 levels): one code per byte, the
# same blockwise statistics, the fused tcgen05 kernel at every M.

def _quant_pair_8bit(N, K, dq, quant_type, seed=0):
    g = synth.generator(seed)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=dq, quant_type=quant_type)
    code = ocb.dynamic_code8() if quant_type == "int8" else ocb.e4m3_code8()
    st = oracle.quantize(w32.numpy(), code, 64, dq, ocb.dynamic_code8(), 256)
    return w, st, g


@pytest.mark.parametrize("quant_type", ["int8", "fp8"])
@pytest.mark.parametrize("N,K,dq", [(256, 512, True), (1000, 1344, False), (3, 100, True)])
def test_8bit_quantize_dequantize_bit_exact(quant_type, N, K, dq):
    w, st, _ = _quant_pair_8bit(N, K, dq, quant_type, seed=N + K)
    assert w.bits == 8 and w.packed.numel() == N * K
    torch.cuda.synchronize()
    _assert_state_equal(w, st)
    f32 = nf4.dequantize(w, torch.float32).cpu().numpy().reshape(-1)
    b16 = bf16_bits(nf4.dequantize(w, torch.bfloat16)).reshape(-1)
    np.testing.assert_array_equal(f32.view(np.uint32), oracle.dequantize(st, "f32").reshape(-1).view(np.uint32))
    np.testing.assert_array_equal(b16, oracle.dequantize(st, "bf16").reshape(-1))


@pytest.mark.parametrize("quant_type", ["int8", "fp8"])
@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (16, 384, 512), (40, 320, 192), (129, 384, 320),
                                   (300, 640, 1024), (700, 640, 1024)])
def test_8bit_fwd_dgrad_parity_and_reruns(quant_type, M, N, K):
    w, st, g = _quant_pair_8bit(N, K, True, quant_type, seed=M + N + K)
    x = synth.activation(M, K, g).to(DEV)
    gy = synth.activation(M, N, g).to(DEV)
    wb = oracle.dequantize(st, "bf16")
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x, w)
    gx = nf4.linear_dgrad(gy, w)
    c = nf4.path_counters()
    assert c["linear_fwd"] == 1 and c["linear_dgrad"] == 1, c
    parity(y, oracle.linear_fwd(bf16_bits(x.cpu()), wb), f"{quant_type} fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy.cpu()), wb), f"{quant_type} dgrad {M}x{N}x{K}")
    for _ in range(3):
        assert torch.equal(nf4.linear_fwd(x, w).view(torch.int16), y.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy, w).view(torch.int16), gx.view(torch.int16))


@pytest.mark.parametrize("quant_type", ["int8", "fp8"])
def test_8bit_identity_probes_exact(quant_type):
    # One-hot rows select single dequantised weights (values; a -0 weight of the
    # e4m3 table sums to +0): the in-kernel 8-bit decode, both operand layouts.
    N, K = 384, 256
    w, st, _ = _quant_pair_8bit(N, K, True, quant_type, seed=9)
    wbf = torch.from_numpy(oracle.dequantize(st, "bf16").view(np.int16)).view(torch.bfloat16).float().numpy()
    eye = torch.eye(K, dtype=torch.bfloat16)
    y = nf4.linear_fwd(eye.to(DEV), w).float().cpu().numpy()
    np.testing.assert_array_equal(y, np.ascontiguousarray(wbf.T))
    eyeN = torch.eye(N, dtype=torch.bfloat16)
    gx = nf4.linear_dgrad(eyeN.to(DEV), w).float().cpu().numpy()
    np.testing.assert_array_equal(gx, wbf)


def test_8bit_stream_k_and_grouped(restore_stream_k):
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    M, N, K = 300, 640, 1024
    w, st, g = _quant_pair_8bit(N, K, True, "int8", seed=21)
    x = synth.activation(M, K, g).to(DEV)
    wb = oracle.dequantize(st, "bf16")
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x, w)
    assert nf4.path_counters()["stream_k"] == 1
    parity(y, oracle.linear_fwd(bf16_bits(x.cpu()), wb), "int8 stream-K fwd")
    ops.set_stream_k(_lib.STREAM_K_AUTO)
    # grouped: 4 experts of 128 rows over one stacked weight, ragged token counts
    E, Ne = 4, 128
    wg, stg, g = _quant_pair_8bit(E * Ne, 256, True, "fp8", seed=22)
    counts = [5, 0, 40, 19]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    xg = synth.activation(T, 256, g)
    gyg = synth.activation(T, Ne, g)
    wbg = oracle.dequantize(stg, "bf16")
    yg = nf4.grouped_fwd(xg.to(DEV), torch.from_numpy(offs).to(DEV), wg, E)
    gxg = nf4.grouped_dgrad(gyg.to(DEV), torch.from_numpy(offs).to(DEV), wg, E)
    xb, gyb = bf16_bits(xg), bf16_bits(gyg)
    yref = np.zeros((T, Ne)); gref = np.zeros((T, 256))
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            yref[r0:r1] = oracle.linear_fwd(xb[r0:r1], wbg[e * Ne:(e + 1) * Ne])
            gref[r0:r1] = oracle.linear_dgrad(gyb[r0:r1], wbg[e * Ne:(e + 1) * Ne])
    parity(yg, yref, "fp8 grouped fwd")
    parity(gxg, gref, "fp8 grouped dgrad")


# ------------------------------------------------------------- fp16 dtype --
# fp16 activations, operand fp16(fp32(code4[q] * scale)) and fp16 outputs: the
# warp-MMA kernels for M <= 16, the fused kernel above.

def _f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (16, 384, 512), (40, 320, 192), (129, 384, 320),
                                   (300, 640, 1024), (700, 640, 1024)])
def test_f16_fwd_dgrad_parity_and_reruns(M, N, K):
    w, st, g = _quant_pair(N, K, True, seed=M + 2 * N + K)
    x = synth.activation(M, K, g).float().half().to(DEV)
    gy = synth.activation(M, N, g).float().half().to(DEV)
    wf = oracle.dequantize_f16(st)
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x, w)
    gx = nf4.linear_dgrad(gy, w)
    c = nf4.path_counters()
    assert y.dtype == torch.float16 and gx.dtype == torch.float16
    if M <= 8:
        assert c["skinny_fwd"] == 1 and c["skinny_dgrad"] == 1, c
    assert c["skinny_fwd"] + c["linear_fwd"] == 1 and c["skinny_dgrad"] + c["linear_dgrad"] == 1, c
    parity(y, oracle.linear_fwd(_f16_bits(x), wf, dtype="f16"), f"f16 fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(_f16_bits(gy), wf, dtype="f16"), f"f16 dgrad {M}x{N}x{K}")
    for _ in range(3):
        assert torch.equal(nf4.linear_fwd(x, w).view(torch.int16), y.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy, w).view(torch.int16), gx.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (3, 136, 1088), (8, 4096, 1024), (9, 520, 2112),
                                   (16, 4096, 4096), (2, 14336, 4096)])
def test_f16_small_m_parity(M, N, K):
    """fp16 products at M <= 16 on the warp-MMA kernels (fp16 MMA, operand
    fp16(fp32(code4[q] * scale)), fp32 accumulation, fixed-order reductions)."""
    w, st, g = _quant_pair(N, K, True, seed=5 * M + N + K)
    x = synth.activation(M, K, g).float().half().to(DEV)
    gy = synth.activation(M, N, g).float().half().to(DEV)
    wf = oracle.dequantize_f16(st)
    nf4.reset_path_counters()
    y = nf4.linear_fwd(x, w)
    gx = nf4.linear_dgrad(gy, w)
    c = nf4.path_counters()
    if M <= 8:
        assert c["skinny_fwd"] == 1 and c["skinny_dgrad"] == 1, c
    assert c["skinny_fwd"] + c["linear_fwd"] == 1 and c["skinny_dgrad"] + c["linear_dgrad"] == 1, c
    assert y.dtype == torch.float16 and gx.dtype == torch.float16
    parity(y, oracle.linear_fwd(_f16_bits(x), wf, dtype="f16"), f"f16 small-M fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(_f16_bits(gy), wf, dtype="f16"), f"f16 small-M dgrad {M}x{N}x{K}")
    assert torch.equal(nf4.linear_fwd(x, w).view(torch.int16), y.view(torch.int16))
    assert torch.equal(nf4.linear_dgrad(gy, w).view(torch.int16), gx.view(torch.int16))


@pytest.mark.parametrize("N,K", [(64, 128), (296, 2048), (4096, 4096)])
def test_f16_small_m_identity_probe_exact(N, K):
    """One-hot fp16 rows read single weight values back through the small-M
    kernels: their operands are exactly the dequantised fp16 weights."""
    w, st, _ = _quant_pair(N, K, True, seed=N + K + 1)
    wf = oracle.dequantize_f16(st)
    nf4.reset_path_counters()
    y = nf4.linear_fwd(torch.eye(K, dtype=torch.float16)[:4].contiguous().to(DEV), w)
    gx = nf4.linear_dgrad(torch.eye(N, dtype=torch.float16)[:4].contiguous().to(DEV), w)
    c = nf4.path_counters()
    assert c["skinny_fwd"] == 1 and c["skinny_dgrad"] == 1, c
    np.testing.assert_array_equal(_f16_bits(y), np.ascontiguousarray(wf.T[:4]))
    np.testing.assert_array_equal(_f16_bits(gx), wf[:4])


def test_f16_identity_probes_exact():
    N, K = 384, 256
    w, st, _ = _quant_pair(N, K, True, seed=31)
    wf = torch.from_numpy(oracle.dequantize_f16(st).view(np.int16)).view(torch.float16).float().numpy()
    y = nf4.linear_fwd(torch.eye(K, dtype=torch.float16, device=DEV), w).float().cpu().numpy()
    np.testing.assert_array_equal(y, np.ascontiguousarray(wf.T))
    gx = nf4.linear_dgrad(torch.eye(N, dtype=torch.float16, device=DEV), w).float().cpu().numpy()
    np.testing.assert_array_equal(gx, wf)


def test_f16_autograd_and_stream_k(restore_stream_k):
    from bit_nf4_quantized_linear_gb300 import autograd
    M, N, K = 300, 640, 1024
    w, st, g = _quant_pair(N, K, True, seed=32)
    wf = oracle.dequantize_f16(st)
    x = synth.activation(M, K, g).float().half().to(DEV).requires_grad_(True)
    gy = synth.activation(M, N, g).float().half().to(DEV)
    y = autograd.nf4_linear(x, w)
    y.backward(gy)
    assert y.dtype == torch.float16 and x.grad.dtype == torch.float16
    parity(y, oracle.linear_fwd(_f16_bits(x), wf, dtype="f16"), "f16 autograd fwd")
    parity(x.grad, oracle.linear_dgrad(_f16_bits(gy), wf, dtype="f16"), "f16 autograd dgrad")
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    nf4.reset_path_counters()
    y2 = nf4.linear_fwd(x.detach(), w)
    assert nf4.path_counters()["stream_k"] == 1
    parity(y2, oracle.linear_fwd(_f16_bits(x), wf, dtype="f16"), "f16 stream-K fwd")


# ------------------------------------------------------ expert epilogues --
# nf4_grouped_fwd_ep: bias, routing-weight row scale and the SwiGLU of interleaved
# gate/up weights fused into the grouped forward, against the oracle's fp64 steps.

def _grouped_ep_case(E, N_e, K, counts, seed, interleave=False):
    g = synth.generator(seed)
    if interleave:
        gate = synth.weight(E * N_e // 2, K, g)
        up = synth.weight(E * N_e // 2, K, g)
        w32 = nf4.interleave_gate_up(gate, up, E)
    else:
        w32 = synth.weight(E * N_e, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    st = oracle.quantize(w32.numpy(), ocb.nf4_code4(), 64, True, ocb.dynamic_code8(), 256)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.activation(int(offs[-1]), K, g)
    return w, st, offs, x, g


@pytest.mark.parametrize("swiglu", [False, True])
def test_grouped_epilogue_bias_scale_swiglu(swiglu):
    E, N_e, K = 4, 256, 320
    counts = [5, 0, 70, 19]
    w, st, offs, x, g = _grouped_ep_case(E, N_e, K, counts, seed=41 + swiglu, interleave=swiglu)
    T = int(offs[-1])
    bias = (torch.randn(E * N_e, generator=g) * 0.1).float()
    scale = torch.rand(T, generator=g).float()
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    y = nf4.grouped_fwd(x.to(DEV), torch.from_numpy(offs).to(DEV), w, E, bias=bias.to(DEV),
                        row_scale=scale.to(DEV), swiglu=swiglu)
    ref = oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, bias=bias.numpy(),
                                      row_scale=scale.numpy(), swiglu=swiglu)
    assert y.shape == (T, N_e // 2 if swiglu else N_e)
    parity(y, ref, f"grouped epilogue swiglu={swiglu}")
    # without the optional parts
    y2 = nf4.grouped_fwd(x.to(DEV), torch.from_numpy(offs).to(DEV), w, E, swiglu=swiglu,
                         bias=None, row_scale=None) if swiglu else None
    if swiglu:
        parity(y2, oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, swiglu=True), "grouped swiglu only")


def test_olmoe_fused_swiglu_and_routing_scale():
    # OLMoE-shaped: 64 experts, hidden 2048, intermediate 1024 (gate and up
    # interleaved: 2048 rows per expert), 512 tokens top-8 (4096 rows).
    E, H, K = 64, 1024, 2048
    g = synth.generator(43)
    _, offs_t = synth.routing(512, E, 8, g)
    offs = offs_t.numpy().astype(np.int32)
    gate = synth.weight(E * H, K, g)
    up = synth.weight(E * H, K, g)
    w32 = nf4.interleave_gate_up(gate, up, E)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    st = oracle.quantize(w32.numpy(), ocb.nf4_code4(), 64, True, ocb.dynamic_code8(), 256)
    T = int(offs[-1])
    x = synth.activation(T, K, g)
    scale = torch.rand(T, generator=g).float()
    y = nf4.grouped_fwd(x.to(DEV), torch.from_numpy(offs).to(DEV), w, E, row_scale=scale.to(DEV),
                        swiglu=True)
    wb = oracle.dequantize(st, "bf16").reshape(E, 2 * H, K)
    ref = oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, row_scale=scale.numpy(), swiglu=True)
    parity(y, ref, "olmoe fused swiglu")


def test_grouped_swiglu_autograd_against_oracle():
    # The backward is one library call; its input gradient and routing-weight
    # gradient are compared with the oracle's grouped_swiglu_dgrad (fp64 steps).
    E, N_e, K = 4, 256, 192
    counts = [9, 40, 0, 23]
    w, st, offs, x, g = _grouped_ep_case(E, N_e, K, counts, seed=44, interleave=True)
    T = int(offs[-1])
    rw = torch.rand(T, generator=g).float()
    gh = synth.activation(T, N_e // 2, g)
    xd = x.to(DEV).requires_grad_(True)
    rwd = rw.to(DEV).requires_grad_(True)
    nf4.reset_path_counters()
    h = nf4.nf4_grouped_swiglu(xd, torch.from_numpy(offs).to(DEV), w, E, row_scale=rwd)
    h.backward(gh.to(DEV))
    c = nf4.path_counters()
    assert c["grouped_fwd"] == 2 and c["grouped_dgrad"] == 1, c
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    parity(h, oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, row_scale=rw.numpy(), swiglu=True),
           "swiglu autograd fwd")
    gx_ref, drw_ref = oracle.grouped_swiglu_dgrad(bf16_bits(x), offs, wb, bf16_bits(gh),
                                                  row_scale=rw.numpy())
    parity(xd.grad, gx_ref, "swiglu autograd dgrad")
    parity(rwd.grad, drw_ref, "swiglu routing-weight grad")


@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_swiglu_bwd_entry_point(with_bias):
    # nf4_grouped_swiglu_bwd through the C ABI: ragged experts (one empty), bias,
    # rows past the last expert untouched in grad_x and zero in the routing-weight
    # gradient, bit-identical reruns.
    E, N_e, K = 3, 384, 256
    counts = [33, 0, 150]
    w, st, offs, x, g = _grouped_ep_case(E, N_e, K, counts, seed=45 + with_bias, interleave=True)
    T = int(offs[-1])
    Tpad = T + 5
    xp = torch.cat([x, synth.activation(5, K, g)])
    rw = torch.rand(Tpad, generator=g).float()
    gh = synth.activation(Tpad, N_e // 2, g)
    bias = (torch.randn(E * N_e, generator=g) * 0.1).float() if with_bias else None
    offs_d = torch.from_numpy(offs).to(DEV)
    outs = []
    for _ in range(2):
        gx, drw = ops.grouped_swiglu_bwd(xp.to(DEV), offs_d, w, E, gh.to(DEV),
                                         bias=None if bias is None else bias.to(DEV),
                                         row_scale=rw.to(DEV), need_row_scale_grad=True)
        outs.append((gx, drw))
    assert torch.equal(outs[0][0].view(torch.int16)[:T], outs[1][0].view(torch.int16)[:T])
    assert torch.equal(outs[0][1], outs[1][1])
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    gx_ref, drw_ref = oracle.grouped_swiglu_dgrad(bf16_bits(x), offs, wb, bf16_bits(gh[:T]),
                                                  bias=None if bias is None else bias.numpy(),
                                                  row_scale=rw[:T].numpy())
    gx, drw = outs[0]
    parity(gx[:T], gx_ref, f"swiglu bwd gx bias={with_bias}")
    parity(drw[:T], drw_ref, f"swiglu bwd drw bias={with_bias}")
    assert torch.count_nonzero(drw[T:]) == 0
    # without the routing-weight gradient, grad_x is the same
    gx2, none = ops.grouped_swiglu_bwd(xp.to(DEV), offs_d, w, E, gh.to(DEV),
                                       bias=None if bias is None else bias.to(DEV),
                                       row_scale=rw.to(DEV))
    assert none is None and torch.equal(gx2.view(torch.int16)[:T], gx.view(torch.int16)[:T])


# ------------------------------------------------------------ fixed token tile --
# The narrower tiles on shapes whose default plan takes 256 tokens (and the
# reverse), and the CTA-pair tile (512 tokens x 256 weight rows on two CTAs, with
# ragged token and column tails and classic splits), through nf4_set_token_tile.

@pytest.fixture
def restore_token_tile():
    yield
    ops.set_token_tile(0)


@pytest.mark.parametrize("bt,M,N,K", [(64, 1100, 640, 1024), (128, 600, 384, 2048), (256, 40, 320, 192),
                                      (64, 513, 256, 8192), (128, 2048, 4096, 4096),
                                      (512, 1100, 640, 1024), (512, 600, 384, 2048), (512, 513, 256, 8192),
                                      (512, 1536, 4096, 4096), (512, 40, 320, 192)])
def test_fixed_token_tile_parity_and_reruns(bt, M, N, K, restore_token_tile):
    ops.set_token_tile(bt)
    sms = nf4.device_check()
    plans = [ops.plan_query(op, M, N, K, sms) for op in (_lib.OP_LINEAR_FWD, _lib.OP_LINEAR_DGRAD)]
    assert all(p["token_tile"] == bt and p["kernel"] == "fused" for p in plans), plans
    w, st, g = _quant_pair(N, K, True, seed=7 * M + N + K)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    rows = _sampled_rows(M, 8) if M * N * K > 2e9 else np.arange(M)
    r = torch.from_numpy(rows).to(DEV)
    parity(y[r], oracle.linear_fwd(bf16_bits(x), wb, rows), f"tile {bt} fwd {M}x{N}x{K}")
    parity(gx[r], oracle.linear_dgrad(bf16_bits(gy), wb, rows), f"tile {bt} dgrad {M}x{N}x{K}")
    for _ in range(2):
        assert torch.equal(nf4.linear_fwd(x.to(DEV), w).view(torch.int16), y.view(torch.int16))
        assert torch.equal(nf4.linear_dgrad(gy.to(DEV), w).view(torch.int16), gx.view(torch.int16))
    assert nf4.device_status() == 0


def test_pair_tiles_identity_probe_and_f16(restore_token_tile):
    # One-hot activations select dequantised weights exactly on CTA-pair tiles
    # (both token halves and both CTAs' rows of every tile); the fp16 dtype on the
    # same tiles within tolerance.
    ops.set_token_tile(512)
    N, K = 384, 1024
    w, st, g = _quant_pair(N, K, True, seed=81)
    wb = oracle.dequantize(st, "bf16")
    y = nf4.linear_fwd(torch.eye(K, dtype=torch.bfloat16, device=DEV), w)
    gx = nf4.linear_dgrad(torch.eye(N, dtype=torch.bfloat16, device=DEV), w)
    np.testing.assert_array_equal(bf16_bits(y), np.ascontiguousarray(wb.T))
    np.testing.assert_array_equal(bf16_bits(gx), wb)
    M = 700
    x = synth.activation(M, K, g).float().half()
    gy = synth.activation(M, N, g).float().half()
    yh = nf4.linear_fwd(x.to(DEV), w)
    gxh = nf4.linear_dgrad(gy.to(DEV), w)
    wh = oracle.dequantize_f16(st)
    parity(yh, oracle.linear_fwd(_f16_bits(x), wh, dtype="f16"), "pair f16 fwd")
    parity(gxh, oracle.linear_dgrad(_f16_bits(gy), wh, dtype="f16"), "pair f16 dgrad")
    assert nf4.device_status() == 0


# ------------------------------------------------------ multi-product launches --
# nf4_linear_fwd_multi / nf4_linear_dgrad_multi: several products of the same M and
# K in one launch, each against the oracle.

def _multi_case(Ns, K, M, seed):
    g = synth.generator(seed)
    ws, sts = [], []
    for N in Ns:
        w32 = synth.weight(N, K, g)
        ws.append(nf4.quantize(w32.to(DEV), double_quant=True))
        sts.append(oracle_state(w32, True))
    x = synth.activation(M, K, g)
    gys = [synth.activation(M, N, g) for N in Ns]
    return ws, sts, x, gys


@pytest.mark.parametrize("M", [1, 40, 300, 513])
@pytest.mark.parametrize("Ns", [(264, 136, 392), (128, 1000), (520,), (96, 384, 1024, 200)])
def test_multi_product_parity(M, Ns):
    K = 320
    ws, sts, x, gys = _multi_case(Ns, K, M, seed=M + sum(Ns))
    nf4.reset_path_counters()
    ys = ops.linear_fwd_multi([x.to(DEV)] * len(Ns), ws)
    gxs = ops.linear_dgrad_multi([gy.to(DEV) for gy in gys], ws)
    c = nf4.path_counters()
    assert c["multi"] == 2 and c["linear_fwd"] == 0 and c["linear_dgrad"] == 0, c
    for p, (N, st) in enumerate(zip(Ns, sts)):
        wb = oracle.dequantize(st, "bf16")
        assert ys[p].shape == (M, N) and gxs[p].shape == (M, K)
        parity(ys[p], oracle.linear_fwd(bf16_bits(x), wb), f"multi fwd p{p} {M}x{N}x{K}")
        parity(gxs[p], oracle.linear_dgrad(bf16_bits(gys[p]), wb), f"multi dgrad p{p} {M}x{N}x{K}")
    ys2 = ops.linear_fwd_multi([x.to(DEV)] * len(Ns), ws)
    gxs2 = ops.linear_dgrad_multi([gy.to(DEV) for gy in gys], ws)
    for a, b in zip(ys + gxs, ys2 + gxs2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_multi_product_llama_qkv_rows():
    # The Llama-3.1-8B q, k, v projections at M = 512 in one launch each way,
    # sampled output rows against the oracle.
    M, K, Ns = 512, 4096, (4096, 1024, 1024)
    ws, sts, x, gys = _multi_case(Ns, K, M, seed=77)
    ys = ops.linear_fwd_multi([x.to(DEV)] * 3, ws)
    gxs = ops.linear_dgrad_multi([gy.to(DEV) for gy in gys], ws)
    rows = np.array([0, 1, 127, 128, 255, 300, 511])
    rows_d = torch.from_numpy(rows).to(DEV)
    for p, st in enumerate(sts):
        wb = oracle.dequantize(st, "bf16")
        parity(ys[p][rows_d], oracle.linear_fwd(bf16_bits(x), wb, rows=rows), f"qkv fwd p{p}")
        parity(gxs[p][rows_d], oracle.linear_dgrad(bf16_bits(gys[p]), wb, rows=rows), f"qkv dgrad p{p}")
    assert nf4.device_status() == 0


def test_multi_product_validation():
    K = 256
    ws, _, x, gys = _multi_case((128, 256), K, 8, seed=5)
    xd = x.to(DEV)
    with pytest.raises(ValueError):
        ops.linear_fwd_multi([xd] * 5, ws * 3)  # more than four products
    w_other, _, _, _ = _multi_case((128,), 320, 8, seed=6)
    with pytest.raises(_lib.NF4Error) as e:  # different K
        ops._multi("nf4_linear_fwd_multi", _lib.lib().nf4_linear_fwd_multi, [xd, xd], [ws[0], w_other[0]],
                   None, lambda w: w.N)
    assert e.value.code == 1
    w8 = nf4.quantize(synth.weight(128, K, synth.generator(7)).to(DEV), double_quant=True, quant_type="int8")
    with pytest.raises(_lib.NF4Error) as e:  # one-byte codes
        ops.linear_fwd_multi([xd, xd], [ws[0], w8])
    assert e.value.code == 7
    y0 = ops.linear_fwd_multi([xd[:0]] * 2, ws)  # M == 0
    assert y0[0].shape == (0, 128)


# ------------------------------------------------------------ top-k combine --
# nf4_moe_combine / nf4_moe_combine_bwd against oracle.moe_combine(_bwd).

def _combine_case(seed, tokens=512, experts=64, topk=8, H=2048):
    g = synth.generator(seed)
    row_token, _ = synth.routing(tokens, experts, topk, g)
    R = row_token.numel()
    rows = synth.activation(R, H, g)
    tr = ops.route_rows(row_token.to(DEV), tokens, topk)
    return rows, tr, g


def test_moe_combine_olmoe_against_oracle():
    rows, tr, g = _combine_case(51)
    nf4.reset_path_counters()
    y = ops.moe_combine(rows.to(DEV), tr)
    assert nf4.path_counters()["moe_combine"] == 1
    tr_h = tr.cpu().numpy()
    assert sorted(tr_h.reshape(-1).tolist()) == list(range(rows.shape[0]))  # each row routed once
    parity(y, oracle.moe_combine(bf16_bits(rows), tr_h), "moe combine")
    assert torch.equal(ops.moe_combine(rows.to(DEV), tr).view(torch.int16), y.view(torch.int16))
    gy = synth.activation(y.shape[0], y.shape[1], g)
    gr = ops.moe_combine_bwd(gy.to(DEV), tr, rows.shape[0])
    np.testing.assert_array_equal(bf16_bits(gr), oracle.moe_combine_bwd(bf16_bits(gy), tr_h, rows.shape[0]))
    assert nf4.device_status() == 0


def test_moe_combine_absent_routes_and_bad_index():
    g = synth.generator(52)
    R, H = 10, 64
    rows = synth.activation(R, H, g)
    tr = torch.tensor([[0, 3, -1], [9, -1, -1], [1, 2, 4]], dtype=torch.int32)
    y = ops.moe_combine(rows.to(DEV), tr.to(DEV))
    parity(y, oracle.moe_combine(bf16_bits(rows), tr.numpy()), "combine with absent routes")
    nf4.device_status(clear=True)
    bad = torch.tensor([[0, 10], [1, 2]], dtype=torch.int32, device=DEV)  # 10 >= R
    y2 = ops.moe_combine(rows.to(DEV), bad)
    assert nf4.device_status(clear=True) == 8  # NF4_ERR_BAD_OFFSETS, the route skipped
    parity(y2[1:], oracle.moe_combine(bf16_bits(rows), bad[1:].cpu().numpy()), "rows with valid routes")


def test_moe_combine_autograd():
    rows, tr, g = _combine_case(53, tokens=64, experts=8, topk=2, H=256)
    rd = rows.to(DEV).requires_grad_(True)
    y = nf4.nf4_combine(rd, tr)
    gy = synth.activation(y.shape[0], y.shape[1], g)
    y.backward(gy.to(DEV))
    tr_h = tr.cpu().numpy()
    parity(y, oracle.moe_combine(bf16_bits(rows), tr_h), "combine fwd")
    np.testing.assert_array_equal(bf16_bits(rd.grad), oracle.moe_combine_bwd(bf16_bits(gy), tr_h, rows.shape[0]))


def test_token_split_at_m8192_rows():
    """M = 8192 at K = N = 4096 runs as CTA-pair tiles over the first 7168 tokens and
    one launch of 256-token tiles over the rest: sampled rows on both sides of the
    boundary and in the tail against the oracle, bit-identical reruns."""
    M, N, K = 8192, 4096, 4096
    assert ops.plan_query(1, M, N, K, 152)["tail_tokens"] == 1024
    w, st, g = _quant_pair(N, K, True, seed=81)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    wb = oracle.dequantize(st, "bf16")
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    rows = np.array([0, 511, 4000, 7166, 7167, 7168, 7169, 7423, 7424, 8000, 8191])
    rows_d = torch.from_numpy(rows).to(DEV)
    parity(y[rows_d], oracle.linear_fwd(bf16_bits(x), wb, rows=rows), "split fwd rows")
    parity(gx[rows_d], oracle.linear_dgrad(bf16_bits(gy), wb, rows=rows), "split dgrad rows")
    assert torch.equal(nf4.linear_fwd(x.to(DEV), w).view(torch.int16), y.view(torch.int16))
    assert nf4.device_status() == 0
