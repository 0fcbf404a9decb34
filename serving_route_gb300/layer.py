"""MegaMoELayer: owns the torch allocations of one layer instance and calls the
C ABI (binding.py).  PyTorch provides device memory and streams only."""
from __future__ import annotations

import torch

from . import binding as B


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class MegaMoELayer:
    def __init__(self, hidden: int, inter: int, num_experts: int, top_k: int, *, max_rows: int,
                 expected_m: int | None = None, capacity_factor: float = 1.0,
                 fuse_fc1: bool = False, check_routes: bool = True, emit_fc1: bool = False,
                 gemm: str = "auto", watchdog_test: bool = False, device="cuda",
                 workspace: torch.Tensor | None = None, gemms: str = "auto",
                 fmt: str = "deepseek", watchdog_route_test: bool = False,
                 swap_ab: bool = True, combine_in_fc2: bool = False):
        """gemm: "auto" (tactic from expected_m), "single" (one CTA per SM) or
        "pair" (CTA pairs, tcgen05 cta_group::2).  swap_ab: forwards of at
        most 64 tokens on single CTAs run the token-as-N GEMMs (False keeps
        the M128 x N256 kernel); combine_in_fc2: on single CTAs (either
        kernel) FC2 folds the combine in (no combine kernel; bit-identical
        output); ignored under CTA pairs.  gemms (fused epilogue only):
        "auto" (FC1 -> FC2 in one persistent launch for short forwards, two
        launches for long ones), "one_launch" or "split"; same results.
        fmt: "deepseek" (1x128 activation / 128x128 weight scales),
        "mxfp8" (one scale per 32 elements along K for both; weights from
        quantize_weights(..., fmt="mxfp8")) or "per_tensor" (one scale per
        expert weight matrix from quantize_weights(..., fmt="per_tensor"),
        and static activation scales given with set_activation_scales).
        workspace: a uint8 device
        tensor shared with other layers whose forwards never overlap with this
        one's (at least workspace_bytes() of every layer that shares it); by
        default the layer allocates its own."""
        self.H, self.I, self.E, self.K = hidden, inter, num_experts, top_k
        assert fmt in ("deepseek", "mxfp8", "per_tensor")
        self.fmt = fmt
        self.max_rows = max_rows
        self.flags = ((B.MOE_FLAG_FUSE_FC1_EPILOGUE if fuse_fc1 else 0)
                      | (B.MOE_FLAG_CHECK_ROUTES if check_routes else 0)
                      | (B.MOE_FLAG_EMIT_FC1 if emit_fc1 else 0)
                      | {"auto": 0, "single": B.MOE_FLAG_GEMM_SINGLE_CTA,
                         "pair": B.MOE_FLAG_GEMM_CTA_PAIR}[gemm]
                      | (B.MOE_FLAG_WATCHDOG_TEST if watchdog_test else 0)
                      | (B.MOE_FLAG_WATCHDOG_ROUTE_TEST if watchdog_route_test else 0)
                      | {"auto": 0, "one_launch": B.MOE_FLAG_GEMMS_ONE_LAUNCH,
                         "split": B.MOE_FLAG_SPLIT_GEMMS}[gemms]
                      | (B.MOE_FLAG_MXFP8 if fmt == "mxfp8" else 0)
                      | (B.MOE_FLAG_PER_TENSOR if fmt == "per_tensor" else 0)
                      | (0 if swap_ab else B.MOE_FLAG_NO_SWAP_AB)
                      | (B.MOE_FLAG_COMBINE_IN_FC2 if combine_in_fc2 else 0))
        em = expected_m if expected_m is not None else max_rows
        ws, wb = B.moe_workspace_query(hidden, inter, num_experts, top_k, self.flags, em, max_rows,
                                       capacity_factor)
        if workspace is None:
            workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        assert workspace.dtype == torch.uint8 and workspace.is_cuda and workspace.is_contiguous()
        assert workspace.numel() >= ws, (workspace.numel(), ws)
        self.workspace = workspace
        self.weight_store = torch.empty(wb, dtype=torch.uint8, device=device)
        self.handle = B.moe_create(hidden, inter, num_experts, top_k, self.flags, em, max_rows,
                                   capacity_factor, self.workspace.data_ptr(), self.workspace.numel(),
                                   self.weight_store.data_ptr(), wb)
        self.out = torch.empty(max_rows, hidden, dtype=torch.bfloat16, device=device)
        B.moe_stage_inputs(self.handle, self.out.data_ptr())

    @staticmethod
    def workspace_bytes(hidden: int, inter: int, num_experts: int, top_k: int, *, max_rows: int,
                        expected_m: int | None = None, capacity_factor: float = 1.0,
                        fuse_fc1: bool = False, emit_fc1: bool = False, gemm: str = "auto",
                        fmt: str = "deepseek") -> int:
        """Workspace size a layer of these dims needs (for a shared workspace)."""
        flags = ((B.MOE_FLAG_FUSE_FC1_EPILOGUE if fuse_fc1 else 0)
                 | (B.MOE_FLAG_EMIT_FC1 if emit_fc1 else 0)
                 | (B.MOE_FLAG_MXFP8 if fmt == "mxfp8" else 0)
                 | (B.MOE_FLAG_PER_TENSOR if fmt == "per_tensor" else 0)
                 | {"auto": 0, "single": B.MOE_FLAG_GEMM_SINGLE_CTA,
                    "pair": B.MOE_FLAG_GEMM_CTA_PAIR}[gemm])
        em = expected_m if expected_m is not None else max_rows
        return B.moe_workspace_query(hidden, inter, num_experts, top_k, flags, em, max_rows,
                                     capacity_factor)[0]

    # -- weights ----------------------------------------------------------------
    @staticmethod
    def quantize_weights(w: torch.Tensor, stream=None, fmt: str = "deepseek"):
        """float32 [n, rows, cols] on the GPU -> (E4M3 uint8, float scales
        [n, rows/128, cols/128]; for fmt="mxfp8" [n, rows, cols/32]; for
        fmt="per_tensor" [n])."""
        assert w.dtype == torch.float32 and w.is_cuda and w.is_contiguous() and w.dim() == 3
        n, r, c = w.shape
        q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        if fmt == "mxfp8":
            s = torch.empty((n, r, c // 32), dtype=torch.float32, device=w.device)
            B.moe_quantize_weights_mx(w.data_ptr(), n, r, c, q.data_ptr(), s.data_ptr(),
                                      _stream_ptr(stream))
        elif fmt == "per_tensor":
            s = torch.empty((n,), dtype=torch.float32, device=w.device)
            B.moe_quantize_weights_pt(w.data_ptr(), n, r, c, q.data_ptr(), s.data_ptr(),
                                      _stream_ptr(stream))
        else:
            assert fmt == "deepseek"
            s = torch.empty((n, r // 128, c // 128), dtype=torch.float32, device=w.device)
            B.moe_quantize_weights(w.data_ptr(), n, r, c, q.data_ptr(), s.data_ptr(),
                                   _stream_ptr(stream))
        return q, s

    @staticmethod
    def requantize_weights_nvfp4(codes: torch.Tensor, block_scales: torch.Tensor,
                                 global_scales: torch.Tensor, stream=None):
        """NVFP4 checkpoint matrices on the GPU -> the default 128x128 FP8
        format (E4M3 uint8 [n, rows, cols], float scales [n, rows/128,
        cols/128]): codes uint8 [n, rows, cols/2] (two E2M1 codes per byte,
        the even column in the low nibble), block_scales uint8 [n, rows,
        cols/16] (E4M3, one per 16 columns), global_scales float32 [n]."""
        for t in (codes, block_scales, global_scales):
            assert t.is_cuda and t.is_contiguous()
        assert codes.dtype == torch.uint8 and block_scales.dtype == torch.uint8
        assert global_scales.dtype == torch.float32 and codes.dim() == 3
        n, r, half = codes.shape
        c = 2 * half
        assert tuple(block_scales.shape) == (n, r, c // 16) and tuple(global_scales.shape) == (n,)
        q = torch.empty((n, r, c), dtype=torch.uint8, device=codes.device)
        s = torch.empty((n, r // 128, c // 128), dtype=torch.float32, device=codes.device)
        B.moe_requantize_weights_nvfp4(codes.data_ptr(), block_scales.data_ptr(),
                                       global_scales.data_ptr(), n, r, c, q.data_ptr(), s.data_ptr(),
                                       _stream_ptr(stream))
        return q, s

    def bind_weights(self, w1_q, w1_s, w2_q, w2_s, stream=None) -> None:
        for t in (w1_q, w1_s, w2_q, w2_s):
            assert t.is_cuda and t.is_contiguous()
        assert tuple(w1_q.shape) == (self.E, 2 * self.I, self.H) and w1_q.dtype == torch.uint8
        assert tuple(w2_q.shape) == (self.E, self.H, self.I) and w2_q.dtype == torch.uint8
        if self.fmt == "mxfp8":
            assert tuple(w1_s.shape) == (self.E, 2 * self.I, self.H // 32)
            assert tuple(w2_s.shape) == (self.E, self.H, self.I // 32)
        elif self.fmt == "per_tensor":
            assert tuple(w1_s.shape) == (self.E,) and tuple(w2_s.shape) == (self.E,)
        else:
            assert tuple(w1_s.shape) == (self.E, 2 * self.I // 128, self.H // 128)
            assert tuple(w2_s.shape) == (self.E, self.H // 128, self.I // 128)
        B.moe_bind_weights(self.handle, w1_q.data_ptr(), w1_s.data_ptr(), w2_q.data_ptr(),
                           w2_s.data_ptr(), _stream_ptr(stream))

    def set_activation_scales(self, x_scale: float, h_scale: float, stream=None) -> None:
        """The static, calibrated activation scales of a per-tensor layer."""
        B.moe_set_activation_scales(self.handle, x_scale, h_scale, _stream_ptr(stream))

    # -- forward ------------------------------------------------------------------
    def stage_output(self, out: torch.Tensor) -> None:
        """Bind another BF16 [max_rows, H] output buffer (moe_stage_inputs); the
        following forwards write there (e.g. two buffers in turn, so the
        device-to-host copy of one forward's output overlaps the next forward)."""
        assert out.dtype == torch.bfloat16 and out.is_cuda and out.is_contiguous()
        assert out.shape[0] >= self.max_rows and out.shape[1] == self.H
        B.moe_stage_inputs(self.handle, out.data_ptr())
        self.out = out

    def forward(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                num_tokens: int | None = None, stream=None) -> torch.Tensor:
        T = x.shape[0] if num_tokens is None else num_tokens
        assert x.dtype == torch.bfloat16 and topk_idx.dtype == torch.int32
        assert topk_w.dtype == torch.float32
        B.moe_forward(self.handle, x.data_ptr(), topk_idx.data_ptr(), topk_w.data_ptr(), T,
                      _stream_ptr(stream))
        return self.out[:T]

    def set_sm_budget(self, max_sms: int) -> None:
        """Cap the SMs the following forwards occupy (0: every SM)."""
        B.moe_set_sm_budget(self.handle, max_sms)

    def read_status(self, stream=None):
        return B.moe_read_status(self.handle, _stream_ptr(stream))

    def set_profile_events(self, events) -> None:
        """torch.cuda.Event objects (created with enable_timing=True); torch
        creates the CUDA event lazily, so each is recorded once here first."""
        if events:
            for e in events:
                e.record()
            torch.cuda.current_stream().synchronize()
        B.moe_set_profile_events(self.handle, [e.cuda_event for e in events] if events else [])

    # -- introspection -------------------------------------------------------------
    def tactic(self) -> dict:
        """The tactic of this layer: CTA pairs or not, GEMM grid, segment padding,
        and the largest ceil(T/512) routed by one cooperative kernel (0: never)."""
        v = B.moe_debug_views(self.handle)
        return dict(gemm_pair=bool(v.gemm_pair), gemm_ctas=int(v.gemm_ctas), pad_rows=int(v.pad_rows),
                    route_coop_blocks=int(v.route_coop_blocks))

    def plan(self, num_tokens: int) -> dict:
        """The kernels a forward of num_tokens tokens enqueues (moe_forward_plan)."""
        p = B.moe_forward_plan(self.handle, num_tokens)
        return dict(route_kernels=p.route_kernels, gemm_launches=p.gemm_launches,
                    swiglu_kernels=p.swiglu_kernels, kernels=p.kernels,
                    swap_ab_tokens=p.swap_ab_tokens, combine_in_fc2=p.combine_in_fc2)

    def route_kernels(self, num_tokens: int) -> int:
        """Kernels the routing step launches for a forward of num_tokens tokens (1 or 3)."""
        return self.plan(num_tokens)["route_kernels"]

    def debug(self) -> dict:
        """torch views of the internal buffers (slices of the workspace); the
        blocked E4M3 buffers a and hq come as row-major copies."""
        v = B.moe_debug_views(self.handle)
        base = self.workspace.data_ptr()
        mx = self.fmt == "mxfp8"
        R = v.rows_alloc
        H, I, E, K = self.H, self.I, self.E, self.K

        def view(ptr, nbytes, dtype, shape):
            off = ptr - base
            t = self.workspace[off:off + nbytes]
            return t.view(dtype).view(shape)

        d = dict(
            status=view(v.status, 4, torch.int32, (1,)),
            counts=view(v.counts, 4 * E, torch.int32, (E,)),
            offsets=view(v.offsets, 4 * (E + 1), torch.int32, (E + 1,)),
            pad_offsets=view(v.pad_offsets, 4 * (E + 1), torch.int32, (E + 1,)),
            perm=view(v.perm, 4 * self.max_rows * K, torch.int32, (self.max_rows * K,)),
            inv=view(v.inv, 4 * self.max_rows * K, torch.int32, (self.max_rows * K,)),
            inv_pad=view(v.inv_pad, 4 * self.max_rows * K, torch.int32, (self.max_rows * K,)),
            a=unblock(view(v.a, R * H, torch.uint8, (R * H,)), R, H),
            a_sf=view(v.a_sf, (R // 128) * kq(H, mx) * 512, torch.uint8, (R // 128, kq(H, mx), 512)),
            hq=unblock(view(v.hq, R * I, torch.uint8, (R * I,)), R, I),
            h_sf=view(v.h_sf, (R // 128) * kq(I, mx) * 512, torch.uint8, (R // 128, kq(I, mx), 512)),
            y=view(v.y, R * H * 2, torch.bfloat16, (R, H)),
            rows_alloc=R,
            gemm_pair=bool(v.gemm_pair),
            gemm_ctas=int(v.gemm_ctas),
            pad_rows=int(v.pad_rows),
        )
        if v.gu:
            d["gu"] = view(v.gu, R * 2 * I * 2, torch.bfloat16, (R, 2 * I))
        return d

    def close(self) -> None:
        if getattr(self, "handle", None):
            B.moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def unblock(flat: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """A blocked E4M3 buffer ([rows/128][cols/128][128][128], every 128x128 block
    contiguous) as a row-major [rows, cols] copy."""
    return flat.view(rows // 128, cols // 128, 128, 128).permute(0, 2, 1, 3).reshape(rows, cols)


def kq(k: int, mx: bool = False) -> int:
    """Scale atoms along a K extent: one per four 128-wide K blocks, or one
    per K block under MXFP8."""
    return k // 128 if mx else (k // 128 + 3) // 4


def sf_atom_rows(atoms: torch.Tensor, rows: int, kblocks: int) -> torch.Tensor:
    """Decode scale atoms [mblocks, kgroups, 512] into E8M0 bytes [rows, kblocks]:
    row r of an m-block, scale unit 4q + j, sits at byte (r%32)*16 + (r//32)*4 + j
    of atom q.  A unit is a 128-wide K block, or under MXFP8 a 32-wide chunk
    (pass kblocks = K/32 then)."""
    mb, kg, _ = atoms.shape
    a = atoms.view(mb, kg, 32, 4, 4)             # [mb, q, r%32, r//32, j]
    a = a.permute(0, 3, 2, 1, 4)                 # [mb, r//32, r%32, q, j]
    return a.reshape(mb * 128, kg * 4)[:rows, :kblocks]
