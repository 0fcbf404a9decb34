"""Shared set-up of the GPU parity tests.

Each side prepares its own inputs from the shared seeded generator:
  * oracle: host generator (C) -> float32 weights -> the oracle's quantiser;
  * GPU:    device generator (CUDA) -> float32 weights in HBM -> the library's
            quantiser (moe_quantize_weights) -> moe_bind_weights.
Routes and x come from the host generator and are copied to the device (they
are inputs, identical on both sides).  No oracle input or expected value is
ever taken from the GPU path.
"""
from __future__ import annotations

import numpy as np
import torch

from gen import inputs as g
from gen import problem
from gen.configs import Workload


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.sqrt(np.sum(b * b))
    return float(np.sqrt(np.sum((a - b) ** 2)) / (den if den > 0 else 1.0))


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return g.bf16_bits_to_f32(bits).astype(np.float64)


def device_weights(wl: Workload, layer_cls, chunk_experts: int = 16, stream=None, fmt="deepseek"):
    """FP32 weights generated on the GPU and quantised there, in expert chunks
    (bounded temporary memory).  Returns (w1q, w1s, w2q, w2s) on the device.
    fmt="mxfp8": scales per row and 32 columns."""
    E, H, I = wl.E, wl.H, wl.I
    dev = torch.device("cuda")
    mx = fmt == "mxfp8"
    pt = fmt == "per_tensor"
    w1q = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
    w1s = torch.empty((E,) if pt else ((E, 2 * I, H // 32) if mx else (E, 2 * I // 128, H // 128)),
                      dtype=torch.float32, device=dev)
    w2q = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
    w2s = torch.empty((E,) if pt else ((E, H, I // 32) if mx else (E, H // 128, I // 128)),
                      dtype=torch.float32, device=dev)
    sp = (stream or torch.cuda.current_stream()).cuda_stream
    n1, n2 = 2 * I * H, H * I
    for e0 in range(0, E, chunk_experts):
        ne = min(chunk_experts, E - e0)
        f1 = torch.empty((ne, 2 * I, H), dtype=torch.float32, device=dev)
        g.dev_normal_f32(wl.seed, g.STREAM_W1, e0 * n1, ne * n1, g.weight_sigma(H), f1.data_ptr(), sp)
        q, s = layer_cls.quantize_weights(f1, stream, fmt=fmt)
        w1q[e0:e0 + ne].copy_(q)
        w1s[e0:e0 + ne].copy_(s)
        del f1, q, s
        f2 = torch.empty((ne, H, I), dtype=torch.float32, device=dev)
        g.dev_normal_f32(wl.seed, g.STREAM_W2, e0 * n2, ne * n2, g.weight_sigma(I), f2.data_ptr(), sp)
        q, s = layer_cls.quantize_weights(f2, stream, fmt=fmt)
        w2q[e0:e0 + ne].copy_(q)
        w2s[e0:e0 + ne].copy_(s)
        del f2, q, s
    return w1q, w1s, w2q, w2s


def oracle_weights(orc, wl: Workload, experts=None, fmt="deepseek"):
    """Oracle-side weights: host generator + the oracle's quantiser.
    experts=None -> all experts; otherwise arrays hold only the listed experts
    in the order given.  fmt="mxfp8": the oracle's MXFP8 quantiser."""
    quant = {"mxfp8": orc.quant_weights_mx, "per_tensor": orc.quant_weights_pt}.get(
        fmt, orc.quant_weights)
    w1q, w1s = quant(problem.w1_f32(wl, experts))
    w2q, w2s = quant(problem.w2_f32(wl, experts))
    return w1q, w1s, w2q, w2s


def host_inputs(wl: Workload):
    x = problem.x_bits(wl)
    idx, w = wl.make_routes()
    return x, idx, w


def to_device(x_bits: np.ndarray, idx: np.ndarray, w: np.ndarray):
    dev = torch.device("cuda")
    xt = torch.from_numpy(x_bits.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    it = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(dev)
    wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(dev)
    return xt, it, wt


def padded_rows(offsets: np.ndarray, pad_offsets: np.ndarray, R: int) -> np.ndarray:
    """GEMM row of every unpadded sorted position p < R."""
    E = len(offsets) - 1
    pos = np.arange(R)
    e = np.searchsorted(offsets, pos, side="right") - 1
    e = np.clip(e, 0, E - 1)
    return pad_offsets[e] + (pos - offsets[e])


def poison_padding(layer) -> int:
    """Writes non-finite values into every padding row of the GEMM segments
    (rows past an expert's routed rows, up to its padded end): E4M3 NaN
    (0x7F) in A and hq, E8M0 NaN (0xFF) in their scale atoms, BF16 NaN in y
    and in gu when it is kept.  Returns the number of padding rows."""
    import serving_route_gb300.binding as B
    d = layer.debug()
    off = d["offsets"].cpu().numpy()
    pad = d["pad_offsets"].cpu().numpy()
    rows = [r for e in range(len(off) - 1) for r in range(pad[e] + off[e + 1] - off[e], pad[e + 1])]
    if not rows:
        return 0
    r = torch.tensor(rows, dtype=torch.long, device="cuda")
    rb, rr = r // 128, r % 128
    v = B.moe_debug_views(layer.handle)
    base, R = layer.workspace.data_ptr(), d["rows_alloc"]
    for ptr, cols in ((v.a, layer.H), (v.hq, layer.I)):
        # blocked [R/128][cols/128][128 rows][128 bytes]
        blk = layer.workspace[ptr - base: ptr - base + R * cols].view(R // 128, cols // 128, 128, 128)
        blk[rb, :, rr, :] = 0x7F
    byte0 = (rr % 32) * 16 + (rr // 32) * 4       # a row's scale bytes in each 512-byte atom
    for sf in (d["a_sf"], d["h_sf"]):
        for j in range(4):
            sf[rb, :, byte0 + j] = 0xFF
    d["y"][r] = float("nan")
    if "gu" in d:
        d["gu"][r] = float("nan")
    torch.cuda.synchronize()
    return len(rows)
