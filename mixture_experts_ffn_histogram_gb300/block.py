"""The MoE expert block as a sequence of libmoe.so calls over caller-owned
device buffers (PyTorch tensors used as plain device memory).

Forward:  moe_route_histogram -> moe_permute -> moe_grouped_gemm_fc1_swiglu
          -> moe_grouped_gemm_fc2 -> moe_combine
Backward: moe_combine_bwd -> moe_grouped_gemm_fc2_bwd (SwiGLU backward fused)
          -> moe_grouped_gemm_fc1_swiglu_bwd -> moe_permute_bwd
"""
from __future__ import annotations

import torch

from . import binding as B

# kernels launched per call sequence (used for the launch count of a step)
FWD_LAUNCHES = 1 + 1 + 1 + 1 + 1     # route (one cooperative kernel), permute, fc1, fc2, combine
BWD_LAUNCHES = 1 + 2 + 2 + 1         # combine_bwd, fc2 dlhs+drhs, fc1 dlhs+drhs, permute_bwd


class MoEBlock:
    def __init__(self, T, D, E, K, F, score_mode=B.SCORE_SOFTMAX_TOPK, train=True,
                 device="cuda"):
        self.d = B.dims(T, D, E, K, F)
        self.T, self.D, self.E, self.K, self.F = T, D, E, K, F
        self.R = T * K
        self.mode = score_mode
        self.train = train
        dev = torch.device(device)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        R = self.R
        self.ids = torch.empty((T, K), dtype=i32, device=dev)
        self.w = torch.empty((T, K), dtype=f32, device=dev)
        self.group_sizes = torch.empty(E, dtype=i32, device=dev)
        self.group_offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.pos = torch.empty((T, K), dtype=i32, device=dev)
        self.row_src = torch.empty(R, dtype=i32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.ws = torch.empty(max(B.moe_workspace_bytes(self.d), 256), dtype=torch.uint8,
                              device=dev)
        self.xs = torch.empty((R, D), dtype=bf, device=dev)
        self.h = torch.empty((R, F), dtype=bf, device=dev)
        self.z = torch.empty((R, 2 * F), dtype=bf, device=dev) if train else None
        self.ys = torch.empty((R, D), dtype=bf, device=dev)
        self.out = torch.empty((T, D), dtype=bf, device=dev)
        if train:
            self.dys = torch.empty((R, D), dtype=bf, device=dev)
            self.dw = torch.empty((T, K), dtype=f32, device=dev)
            self.dz = torch.empty((R, 2 * F), dtype=bf, device=dev)
            self.dwo = torch.empty((E, F, D), dtype=bf, device=dev)
            self.dxs = torch.empty((R, D), dtype=bf, device=dev)
            self.dwi = torch.empty((E, D, 2 * F), dtype=bf, device=dev)
            self.dx = torch.empty((T, D), dtype=bf, device=dev)

    def forward_fused(self, x, wi, wo, logits=None, bias=None, ids=None, w=None, stream=None):
        """The inference forward through moe_fused_forward: routing, then FC1
        on rows gathered straight from x and FC2 with the weighted combine in
        its epilogue (no xs, no ys).  Needs a whole wi; h and an fp32 [T, D]
        accumulator are the block's scratch."""
        d = self.d
        self._check_weights(wi, wo)
        if isinstance(wi, (list, tuple)):
            raise ValueError("the fused forward takes a whole wi")
        if self.mode == B.SCORE_GIVEN:
            self.ids.copy_(ids)
            self.w.copy_(w)
        if getattr(self, "acc", None) is None:
            self.acc = torch.empty((self.T, self.D), dtype=torch.float32, device=self.out.device)
        B.moe_route_histogram(logits, bias, self.mode, self.ids, self.w, self.group_sizes,
                              self.group_offsets, self.pos, self.row_src, self.status, self.ws,
                              d, stream)
        B.moe_fused_forward(x, self.w, self.row_src, self.group_offsets, wi, wo, self.h, self.acc,
                            self.out, self.status, self.ws, d, stream)
        return self.out

    def _check_weights(self, wi, wo):
        """The library builds its tensor maps from the block's dims, so a
        weight of another shape or dtype would be read (and its gradient
        written) out of bounds: reject it before any launch."""
        D, F, E = self.D, self.F, self.E
        if wo.dtype != torch.bfloat16 or tuple(wo.shape) != (E, F, D):
            raise ValueError(f"wo must be bf16 [{E}, {F}, {D}], got {wo.dtype} {tuple(wo.shape)}")
        if isinstance(wi, (list, tuple)):
            self._ranges(wi)
        elif wi.dtype != torch.bfloat16 or tuple(wi.shape) != (E, D, 2 * F):
            raise ValueError(f"wi must be bf16 [{E}, {D}, {2 * F}], got {wi.dtype} "
                             f"{tuple(wi.shape)}")

    def forward(self, x, wi, wo, logits=None, bias=None, ids=None, w=None, stream=None):
        d = self.d
        self._check_weights(wi, wo)
        if self.mode == B.SCORE_GIVEN:
            self.ids.copy_(ids)
            self.w.copy_(w)
        B.moe_route_histogram(logits, bias, self.mode, self.ids, self.w, self.group_sizes,
                              self.group_offsets, self.pos, self.row_src, self.status, self.ws,
                              d, stream)
        B.moe_permute(x, self.pos, self.xs, d, stream)
        if isinstance(wi, (list, tuple)):
            # split-expert layout: wi as expert-range buffers, FC1 as chained
            # grouped GEMM calls into the one h (and z)
            for e0, e1, part in self._ranges(wi):
                B.moe_grouped_gemm_fc1_swiglu_experts(self.xs, part, self.group_offsets, e0, e1,
                                                      self.h, self.z, self.status, self.ws, d,
                                                      stream)
        else:
            B.moe_grouped_gemm_fc1_swiglu(self.xs, wi, self.group_offsets, self.h, self.z,
                                          self.status, self.ws, d, stream)
        B.moe_grouped_gemm_fc2(self.h, wo, self.group_offsets, self.ys, self.status, self.ws, d,
                               stream)
        B.moe_combine(self.ys, self.w, self.pos, self.out, d, stream)
        return self.out

    def backward(self, dy, wi, wo, stream=None):
        d = self.d
        self._check_weights(wi, wo)
        B.moe_combine_bwd(dy, self.ys, self.w, self.pos, self.dys, self.dw, d, stream)
        B.moe_grouped_gemm_fc2_bwd(self.dys, self.h, wo, self.z, self.group_offsets, self.dz,
                                   self.dwo, self.status, self.ws, d, stream)
        if isinstance(wi, (list, tuple)):
            # split-expert layout: dxs chained over the ranges; dwi_parts[i]
            # is the gradient of wi[i]
            if getattr(self, "dwi_parts", None) is None or \
                    [p.shape for p in self.dwi_parts] != [p.shape for p in wi]:
                self.dwi_parts = [torch.empty_like(p) for p in wi]
            for (e0, e1, part), dpart in zip(self._ranges(wi), self.dwi_parts):
                B.moe_grouped_gemm_fc1_bwd_experts(self.dz, self.xs, part, self.group_offsets, e0,
                                                   e1, self.dxs, dpart, self.status, self.ws, d,
                                                   stream)
        else:
            B.moe_grouped_gemm_fc1_swiglu_bwd(self.dz, None, self.xs, wi, self.group_offsets,
                                              self.dxs, self.dwi, self.status, self.ws, d, stream)
        B.moe_permute_bwd(self.dxs, self.pos, self.dx, d, stream)
        return self.dx

    def _ranges(self, parts):
        """(e_begin, e_end, tensor) of each expert-range buffer of a split wi."""
        out, e0 = [], 0
        for part in parts:
            if part.dtype != torch.bfloat16 or part.dim() != 3 or \
                    tuple(part.shape[1:]) != (self.D, 2 * self.F):
                raise ValueError(f"each wi part must be bf16 [experts, {self.D}, {2 * self.F}], "
                                 f"got {part.dtype} {tuple(part.shape)}")
            e1 = e0 + int(part.shape[0])
            out.append((e0, e1, part))
            e0 = e1
        if e0 != self.E:
            raise ValueError(f"the wi parts cover {e0} experts, the block has {self.E}")
        return out


class MoEBlockMX:
    """The block in MXFP8.  ``set_weights`` quantizes the expert weights (for
    the forward, and with ``train`` also along their other axis for the
    dgrads); each ``forward`` routes, quantizes the tokens while permuting
    them, runs FC1 + SwiGLU and FC2 on the tensor cores' block-scaled MMA (h
    quantized in FC1's epilogue; with ``train`` also h and z in bf16) and
    combines.  ``backward`` (train only): combine backward, the gradient
    quantized along D and along tokens, the FC2 dgrad with the SwiGLU
    backward and the dwo wgrad, dz quantized along 2F and along tokens, x
    quantized along tokens straight from its token-major rows, the FC1
    dgrad and the dwi wgrad, and the permute backward.  Every buffer is
    allocated once, in the library's MX layouts.

    ``wgrad="bf16"`` keeps the two weight gradients in bf16: the forward
    also writes the sorted rows xs in bf16, and dwo = h^T dys, dwi = xs^T dz
    run on the bf16 grouped GEMM, so no operand is quantized along tokens
    (the forward and both dgrads stay in MXFP8)."""

    def __init__(self, T, D, E, K, F, score_mode=B.SCORE_SOFTMAX_TOPK, device="cuda",
                 train=False, wgrad="mx"):
        if wgrad not in ("mx", "bf16"):
            raise ValueError(f"wgrad must be 'mx' or 'bf16', got {wgrad!r}")
        self.d = d = B.dims(T, D, E, K, F)
        self.T, self.D, self.E, self.K, self.F = T, D, E, K, F
        self.R = R = T * K
        self.mode = score_mode
        self.train = train
        self.wgrad = wgrad
        dev = torch.device(device)
        i32, bf = torch.int32, torch.bfloat16

        def u8(which):
            return torch.empty(max(B.moe_mx_bytes(d, which), 16), dtype=torch.uint8, device=dev)

        self.ids = torch.empty((T, K), dtype=i32, device=dev)
        self.w = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.group_sizes = torch.empty(E, dtype=i32, device=dev)
        self.group_offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.pos = torch.empty((T, K), dtype=i32, device=dev)
        self.row_src = torch.empty(R, dtype=i32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.ws = torch.empty(max(B.moe_workspace_bytes(d), 256), dtype=torch.uint8, device=dev)
        self.wiq, self.wisc = u8(B.MX_WIQ), u8(B.MX_WISC)
        self.woq, self.wosc = u8(B.MX_WOQ), u8(B.MX_WOSC)
        self.xq, self.xsc = u8(B.MX_XQ), u8(B.MX_XSC)
        self.hq, self.hsc = u8(B.MX_HQ), u8(B.MX_HSC)
        self.ys = torch.empty((R, D), dtype=bf, device=dev)
        self.out = torch.empty((T, D), dtype=bf, device=dev)
        if train:
            self.h = torch.empty((R, F), dtype=bf, device=dev)
            self.z = torch.empty((R, 2 * F), dtype=bf, device=dev)
            self.dys = torch.empty((R, D), dtype=bf, device=dev)
            self.dw = torch.empty((T, K), dtype=torch.float32, device=dev)
            self.dz = torch.empty((R, 2 * F), dtype=bf, device=dev)
            self.dxs = torch.empty((R, D), dtype=bf, device=dev)
            self.dx = torch.empty((T, D), dtype=bf, device=dev)
            self.dwi = torch.empty((E, D, 2 * F), dtype=bf, device=dev)
            self.dwo = torch.empty((E, F, D), dtype=bf, device=dev)
            self.wiq_b, self.wisc_b = u8(B.MX_WIQ_BWD), u8(B.MX_WISC_BWD)
            self.woq_b, self.wosc_b = u8(B.MX_WOQ_BWD), u8(B.MX_WOSC_BWD)
            self.dyq, self.dysc = u8(B.MX_DYQ), u8(B.MX_DYSC)
            self.dzq, self.dzsc = u8(B.MX_DZQ), u8(B.MX_DZSC)
            if wgrad == "mx":
                self.xt, self.xtsc = u8(B.MX_XT), u8(B.MX_XTSC)
                self.ht, self.htsc = u8(B.MX_HT), u8(B.MX_HTSC)
                self.dyt, self.dytsc = u8(B.MX_DYT), u8(B.MX_DYTSC)
                self.dzt, self.dztsc = u8(B.MX_DZT), u8(B.MX_DZTSC)
            else:
                self.xs = torch.empty((R, D), dtype=bf, device=dev)
        self.x = None

    def set_weights(self, wi, wo, stream=None):
        tr = self.train
        B.moe_mx_quantize_wi(wi, self.wiq, self.wisc, self.d, stream,
                             wq_bwd=self.wiq_b if tr else None, wsc_bwd=self.wisc_b if tr else None)
        B.moe_mx_quantize_wo(wo, self.woq, self.wosc, self.d, stream,
                             wq_bwd=self.woq_b if tr else None, wsc_bwd=self.wosc_b if tr else None)

    def forward(self, x, logits=None, bias=None, ids=None, w=None, stream=None):
        d = self.d
        if self.mode == B.SCORE_GIVEN:
            self.ids.copy_(ids)
            self.w.copy_(w)
        B.moe_route_histogram(logits, bias, self.mode, self.ids, self.w, self.group_sizes,
                              self.group_offsets, self.pos, self.row_src, self.status, self.ws,
                              d, stream)
        B.moe_mx_permute_quantize(x, self.pos, self.group_offsets, self.xq, self.xsc, d, stream)
        if self.train and self.wgrad == "bf16":
            B.moe_permute(x, self.pos, self.xs, d, stream)
        B.moe_mx_grouped_gemm_fc1_swiglu(self.xq, self.xsc, self.wiq, self.wisc,
                                         self.group_offsets, self.hq, self.hsc,
                                         self.h if self.train else None, self.status, d, stream,
                                         z=self.z if self.train else None)
        B.moe_mx_grouped_gemm_fc2(self.hq, self.hsc, self.woq, self.wosc, self.group_offsets,
                                  self.ys, self.status, d, stream)
        B.moe_combine(self.ys, self.w, self.pos, self.out, d, stream)
        self.x = x
        return self.out

    def backward(self, dy, stream=None):
        if not self.train:
            raise RuntimeError("the block was built without train=True")
        if self.x is None:
            raise RuntimeError("backward needs a forward first")
        d, D, F = self.d, self.D, self.F
        offs = self.group_offsets
        B.moe_mx_combine_bwd(dy, self.ys, self.w, self.pos, offs, self.dys, self.dyq, self.dysc,
                             self.dw, d, stream)
        if self.wgrad == "bf16":
            B.moe_mx_grouped_gemm_fc2_bwd(self.dyq, self.dysc, self.woq_b, self.wosc_b, self.z,
                                          None, None, None, None, offs, self.dz, None,
                                          self.status, d, stream)
            B.moe_grouped_gemm_fc2_bwd(self.dys, self.h, None, None, offs, None, self.dwo,
                                       self.status, self.ws, d, stream)
            B.moe_mx_quantize_rows(self.dz, 2 * F, offs, self.dzq, self.dzsc, d, stream)
            B.moe_mx_grouped_gemm_fc1_bwd(self.dzq, self.dzsc, self.wiq_b, self.wisc_b, None,
                                          None, None, None, offs, self.dxs, None, self.status,
                                          d, stream)
            B.moe_grouped_gemm_fc1_swiglu_bwd(self.dz, None, self.xs, None, offs, None, self.dwi,
                                              self.status, self.ws, d, stream)
            B.moe_permute_bwd(self.dxs, self.pos, self.dx, d, stream)
            return self.dx
        B.moe_mx_quantize_tokens(self.dys, None, D, offs, self.dyt, self.dytsc, d, stream)
        B.moe_mx_quantize_tokens(self.h, None, F, offs, self.ht, self.htsc, d, stream)
        B.moe_mx_grouped_gemm_fc2_bwd(self.dyq, self.dysc, self.woq_b, self.wosc_b, self.z,
                                      self.ht, self.htsc, self.dyt, self.dytsc, offs, self.dz,
                                      self.dwo, self.status, d, stream)
        B.moe_mx_quantize_rows(self.dz, 2 * F, offs, self.dzq, self.dzsc, d, stream)
        B.moe_mx_quantize_tokens(self.dz, None, 2 * F, offs, self.dzt, self.dztsc, d, stream)
        B.moe_mx_quantize_tokens(self.x, self.row_src, D, offs, self.xt, self.xtsc, d, stream)
        B.moe_mx_grouped_gemm_fc1_bwd(self.dzq, self.dzsc, self.wiq_b, self.wisc_b, self.xt,
                                      self.xtsc, self.dzt, self.dztsc, offs, self.dxs, self.dwi,
                                      self.status, d, stream)
        B.moe_permute_bwd(self.dxs, self.pos, self.dx, d, stream)
        return self.dx


class HostPipeline:
    """Steps of a MoEBlock (fwd+bwd when the block trains, else forward only)
    whose per-step activations live in pinned host memory, with the
    host<->device copies overlapped with the kernels.

    Step i's inputs (x, dy, and logits or ids/w) go up on an upload stream
    into one of two device slots while step i-1 computes; step i's `out` goes
    down on a download stream while its backward (or step i+1) runs, and its
    `dx` while step i+1 runs.  Ordering comes from CUDA events only (no host
    sync):
    - an upload into a slot waits until the step that last used it is done;
    - a step waits for its upload; `out` and `dx` alternate between two
      device buffers, and a step's forward (backward) waits only until the
      download of the `out` (`dx`) two steps back has read the buffer it
      reuses (with one buffer each, a backward waited for the previous
      step's whole `dx` download, which starts only when that step ends).
    Every step still moves all of its bytes across the host link; only the
    waiting is hidden.  `synchronize()` waits for the last download.
    """

    def __init__(self, blk: MoEBlock, wi, wo, bias=None):
        self.blk, self.wi, self.wo, self.bias = blk, wi, wo, bias
        self.train = blk.train
        dev = blk.out.device
        self.compute = torch.cuda.Stream(dev)
        self.up = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        T, D, E, K = blk.T, blk.D, blk.E, blk.K
        given = blk.mode == B.SCORE_GIVEN
        self.slots = []
        for _ in range(2):
            self.slots.append({
                "x": torch.empty((T, D), dtype=torch.bfloat16, device=dev),
                "dy": torch.empty((T, D), dtype=torch.bfloat16, device=dev) if self.train else None,
                "logits": None if given else torch.empty((T, E), dtype=torch.float32, device=dev),
                "ids": torch.empty((T, K), dtype=torch.int32, device=dev) if given else None,
                "w": torch.empty((T, K), dtype=torch.float32, device=dev) if given else None,
            })
        self.outs = [blk.out, torch.empty_like(blk.out)]
        self.dxs = [blk.dx, torch.empty_like(blk.dx)] if self.train else [None, None]
        self.slot_free = [None, None]   # event: the last step using the slot is done
        self.out_read = [None, None]    # event: the download of outs[k] has read it
        self.dx_read = [None, None]     # event: the download of dxs[k] has read it
        self.i = 0

    def step(self, x_h, out_h, dy_h=None, dx_h=None, logits_h=None, ids_h=None, w_h=None):
        """Queues one step: inputs from the pinned host tensors, `out` (and,
        training, `dx`) into the pinned host tensors `out_h` (`dx_h`), valid
        after the next synchronize()."""
        blk, k = self.blk, self.i % 2
        s = self.slots[k]
        with torch.cuda.stream(self.up):
            if self.slot_free[k] is not None:
                self.up.wait_event(self.slot_free[k])
            s["x"].copy_(x_h, non_blocking=True)
            if self.train:
                s["dy"].copy_(dy_h, non_blocking=True)
            if s["logits"] is not None:
                s["logits"].copy_(logits_h, non_blocking=True)
            else:
                s["ids"].copy_(ids_h, non_blocking=True)
                s["w"].copy_(w_h, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(self.up)
        out, dx = self.outs[k], self.dxs[k]
        blk.out = out
        if self.train:
            blk.dx = dx
        with torch.cuda.stream(self.compute):
            self.compute.wait_event(uploaded)
            if self.out_read[k] is not None:
                self.compute.wait_event(self.out_read[k])
            blk.forward(s["x"], self.wi, self.wo, logits=s["logits"], bias=self.bias,
                        ids=s["ids"], w=s["w"])
            fwd_done = torch.cuda.Event()
            fwd_done.record(self.compute)
            done = fwd_done
            if self.train:
                if self.dx_read[k] is not None:
                    self.compute.wait_event(self.dx_read[k])
                blk.backward(s["dy"], self.wi, self.wo)
                done = torch.cuda.Event()
                done.record(self.compute)
        self.slot_free[k] = done
        with torch.cuda.stream(self.down):
            self.down.wait_event(fwd_done)
            out_h.copy_(out, non_blocking=True)
            self.out_read[k] = torch.cuda.Event()
            self.out_read[k].record(self.down)
            if self.train:
                self.down.wait_event(done)
                dx_h.copy_(dx, non_blocking=True)
                self.dx_read[k] = torch.cuda.Event()
                self.dx_read[k].record(self.down)
        self.i += 1

    def synchronize(self):
        self.down.synchronize()
        self.compute.synchronize()


class GraphStep:
    """One step of a MoEBlock (forward, plus backward when `dy` is given)
    captured once into a CUDA graph and replayed with `replay()`.

    The graph holds the block's launches with the device addresses of the
    tensors passed here, so a caller feeds new data by writing into those
    same tensors (x, logits or ids/w, dy) before each replay; outputs land in
    the block's buffers (blk.out, blk.dx, ...).  Replaying one graph costs
    one launch on the host instead of one per kernel, which is what small
    steps (a few thousand tokens) are bound by.  The constructor runs the
    step once uncaptured first, so that the library's once-per-process setup
    (SM count, driver entry point, occupancy queries) happens outside the
    capture.
    """

    def __init__(self, blk: MoEBlock, x, wi, wo, logits=None, bias=None, ids=None, w=None,
                 dy=None):
        self.blk = blk
        self.args = (x, wi, wo, logits, bias, ids, w, dy)
        side = torch.cuda.Stream(blk.out.device)
        side.wait_stream(torch.cuda.current_stream(blk.out.device))
        with torch.cuda.stream(side):
            self._run()
        torch.cuda.current_stream(blk.out.device).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._run()

    def _run(self):
        x, wi, wo, logits, bias, ids, w, dy = self.args
        self.blk.forward(x, wi, wo, logits=logits, bias=bias, ids=ids, w=w)
        if dy is not None:
            self.blk.backward(dy, wi, wo)

    def replay(self):
        self.graph.replay()
