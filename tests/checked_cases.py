"""Every product path of the library on small, ragged shapes, run against the
checked debug build (in-kernel index checks; started with NF4_CHECKED=1 by
tests/test_gpu_checked.py, in a process of its own because the binding loads one
library per process).  Each result is compared with the CPU oracle; at the end
the device status word must be clean, and the injected failure of the index
check must show as NF4_ERR_BOUNDS.  Prints one line per case and exits non-zero
on the first failure."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from oracle import codebooks as ocb  # noqa: E402
import bit_nf4_quantized_linear_gb300 as nf4  # noqa: E402
from bit_nf4_quantized_linear_gb300 import _lib, ops, synth  # noqa: E402
from tests.helpers import bf16_bits, oracle_state, parity  # noqa: E402

DEV = torch.device("cuda:0")


def f16_bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def status_clean(what):
    torch.cuda.synchronize()
    s = nf4.device_status(clear=True)
    assert s == 0, f"{what}: device status {_lib.STATUS_NAMES.get(s, s)}"


def dense(M, N, K, dq=True, seed=0, what="", f16=False, quant_type="nf4"):
    g = synth.generator(seed)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=dq, quant_type=quant_type)
    if quant_type == "nf4":
        st = oracle_state(w32, dq)
    else:
        st = oracle.quantize(w32.numpy(), ocb.dynamic_code8(), 64, dq, ocb.dynamic_code8(), 256)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    if f16:
        x, gy = x.float().half(), gy.float().half()
        wf = oracle.dequantize_f16(st)
        y = nf4.linear_fwd(x.to(DEV), w)
        gx = nf4.linear_dgrad(gy.to(DEV), w)
        parity(y, oracle.linear_fwd(f16_bits(x), wf, dtype="f16"), f"{what} fwd")
        parity(gx, oracle.linear_dgrad(f16_bits(gy), wf, dtype="f16"), f"{what} dgrad")
    else:
        wb = oracle.dequantize(st, "bf16")
        y = nf4.linear_fwd(x.to(DEV), w)
        gx = nf4.linear_dgrad(gy.to(DEV), w)
        parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"{what} fwd")
        parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"{what} dgrad")
    status_clean(what)
    print("ok", what, M, N, K, flush=True)


def grouped(seed=0):
    E, N_e, K = 6, 192, 256
    g = synth.generator(seed)
    w32 = synth.weight(E * N_e, K, g)
    row_token, offsets = synth.routing(50, E, 2, g)
    x = synth.activation(50, K, g)[row_token].contiguous()
    T = x.shape[0]
    gy = synth.activation(T, N_e, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    wb = oracle.dequantize(oracle_state(w32, True), "bf16").reshape(E, N_e, K)
    offs = offsets.numpy()
    y = nf4.grouped_fwd(x.to(DEV), offsets.to(DEV), w, E)
    gx = nf4.grouped_dgrad(gy.to(DEV), offsets.to(DEV), w, E)
    parity(y, oracle.grouped_fwd(bf16_bits(x), offs, wb), "grouped fwd")
    parity(gx, oracle.grouped_dgrad(bf16_bits(gy), offs, wb), "grouped dgrad")
    status_clean("grouped")
    print("ok grouped", flush=True)


def grouped_swiglu(seed=0):
    E, N_e, K = 3, 256, 192
    counts = [9, 0, 40]
    g = synth.generator(seed)
    gate = synth.weight(E * N_e // 2, K, g)
    up = synth.weight(E * N_e // 2, K, g)
    w32 = nf4.interleave_gate_up(gate, up, E)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    st = oracle.quantize(w32.numpy(), ocb.nf4_code4(), 64, True, ocb.dynamic_code8(), 256)
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    x = synth.activation(T, K, g)
    rw = torch.rand(T, generator=g).float()
    bias = (torch.randn(E * N_e, generator=g) * 0.1).float()
    gh = synth.activation(T, N_e // 2, g)
    offs_d = torch.from_numpy(offs).to(DEV)
    h = nf4.grouped_fwd(x.to(DEV), offs_d, w, E, bias=bias.to(DEV), row_scale=rw.to(DEV), swiglu=True)
    parity(h, oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, bias=bias.numpy(), row_scale=rw.numpy(),
                                          swiglu=True), "grouped swiglu fwd")
    gx, drw = ops.grouped_swiglu_bwd(x.to(DEV), offs_d, w, E, gh.to(DEV), bias=bias.to(DEV),
                                     row_scale=rw.to(DEV), need_row_scale_grad=True)
    gx_ref, drw_ref = oracle.grouped_swiglu_dgrad(bf16_bits(x), offs, wb, bf16_bits(gh), bias=bias.numpy(),
                                                  row_scale=rw.numpy())
    parity(gx, gx_ref, "grouped swiglu bwd grad_x")
    parity(drw, drw_ref, "grouped swiglu bwd routing-weight grad")
    status_clean("grouped swiglu")
    print("ok grouped swiglu", flush=True)


def multi(seed=0):
    K, M, Ns = 320, 300, (264, 136, 392)
    g = synth.generator(seed)
    ws, wbs = [], []
    for N in Ns:
        w32 = synth.weight(N, K, g)
        ws.append(nf4.quantize(w32.to(DEV), double_quant=True))
        wbs.append(oracle.dequantize(oracle_state(w32, True), "bf16"))
    x = synth.activation(M, K, g)
    gys = [synth.activation(M, N, g) for N in Ns]
    ys = ops.linear_fwd_multi([x.to(DEV)] * len(Ns), ws)
    gxs = ops.linear_dgrad_multi([gy.to(DEV) for gy in gys], ws)
    for p, wb in enumerate(wbs):
        parity(ys[p], oracle.linear_fwd(bf16_bits(x), wb), f"multi fwd p{p}")
        parity(gxs[p], oracle.linear_dgrad(bf16_bits(gys[p]), wb), f"multi dgrad p{p}")
    status_clean("multi")
    print("ok multi", flush=True)


def combine(seed=0):
    g = synth.generator(seed)
    row_token, _ = synth.routing(64, 8, 2, g)
    R = row_token.numel()
    rows = synth.activation(R, 256, g)
    tr = ops.route_rows(row_token.to(DEV), 64, 2)
    y = ops.moe_combine(rows.to(DEV), tr)
    parity(y, oracle.moe_combine(bf16_bits(rows), tr.cpu().numpy()), "combine")
    gy = synth.activation(64, 256, g)
    gr = ops.moe_combine_bwd(gy.to(DEV), tr, R)
    assert np.array_equal(bf16_bits(gr), oracle.moe_combine_bwd(bf16_bits(gy), tr.cpu().numpy(), R))
    status_clean("combine")
    print("ok combine", flush=True)


def main():
    assert _lib.checked_build(), "NF4_CHECKED=1 must load the checked build"
    nf4.device_status(clear=True)
    # default plans: small-M kernels, tiles, cluster splits, stream-K
    for i, (M, N, K) in enumerate([(1, 200, 320), (3, 136, 1088), (8, 96, 5120), (9, 520, 2112),
                                   (17, 264, 320), (100, 296, 640), (300, 640, 1024), (700, 384, 512)]):
        dense(M, N, K, dq=bool(i % 2), seed=i, what="auto")
    # forced schedules and paths
    ops.set_small_m_path(_lib.SMALL_M_SIMT)
    dense(3, 264, 320, seed=20, what="simt gemv")
    ops.set_small_m_path(_lib.SMALL_M_TILES)
    dense(5, 264, 320, seed=21, what="small-M tiles")
    ops.set_small_m_path(_lib.SMALL_M_AUTO)
    ops.set_stream_k(_lib.STREAM_K_FORCE)
    dense(200, 392, 576, seed=22, what="stream-K")
    ops.set_stream_k(_lib.STREAM_K_AUTO)
    ops.set_cluster_split(_lib.CLUSTER_SPLIT_FORCE)
    dense(128, 512, 1024, seed=23, what="cluster split")
    ops.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)
    for bt, M in ((16, 40), (32, 70), (64, 130), (128, 200), (256, 300), (512, 600)):
        ops.set_token_tile(bt)
        dense(M, 264, 320, seed=30 + bt, what=f"token tile {bt}")
    ops.set_token_tile(0)
    # dtypes and code widths
    for M in (1, 16, 300):
        dense(M, 264, 320, seed=40 + M, what="fp16", f16=True)
    for M in (3, 200):
        dense(M, 264, 320, seed=50 + M, what="8-bit codes", quant_type="int8")
    grouped(seed=60)
    grouped_swiglu(seed=61)
    multi(seed=62)
    combine(seed=63)
    # the check itself: a failure injected into the next fused launch's index checks
    # is recorded (its loads are skipped), and the next launch is clean again
    _lib.inject_bounds_failure()
    g = synth.generator(70)
    w = nf4.quantize(synth.weight(264, 320, g).to(DEV), double_quant=True)
    nf4.linear_fwd(synth.activation(40, 320, g).to(DEV), w)
    torch.cuda.synchronize()
    s = nf4.device_status(clear=True)
    assert s == 9, f"injected index-check failure: device status {s}, expected NF4_ERR_BOUNDS"
    print("ok injected failure recorded", flush=True)
    dense(40, 264, 320, seed=71, what="after injection")
    print("CHECKED OK", flush=True)


if __name__ == "__main__":
    main()
