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
FWD_LAUNCHES = 3 + 1 + 1 + 1 + 1     # route(topk+hist, scan, rank), permute, fc1, fc2, combine
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

    def forward(self, x, wi, wo, logits=None, bias=None, ids=None, w=None, stream=None):
        d = self.d
        if self.mode == B.SCORE_GIVEN:
            self.ids.copy_(ids)
            self.w.copy_(w)
        B.moe_route_histogram(logits, bias, self.mode, self.ids, self.w, self.group_sizes,
                              self.group_offsets, self.pos, self.row_src, self.status, self.ws,
                              d, stream)
        B.moe_permute(x, self.pos, self.xs, d, stream)
        B.moe_grouped_gemm_fc1_swiglu(self.xs, wi, self.group_offsets, self.h, self.z,
                                      self.status, self.ws, d, stream)
        B.moe_grouped_gemm_fc2(self.h, wo, self.group_offsets, self.ys, self.status, self.ws, d,
                               stream)
        B.moe_combine(self.ys, self.w, self.pos, self.out, d, stream)
        return self.out

    def backward(self, dy, wi, wo, stream=None):
        d = self.d
        B.moe_combine_bwd(dy, self.ys, self.w, self.pos, self.dys, self.dw, d, stream)
        B.moe_grouped_gemm_fc2_bwd(self.dys, self.h, wo, self.z, self.group_offsets, self.dz,
                                   self.dwo, self.status, self.ws, d, stream)
        B.moe_grouped_gemm_fc1_swiglu_bwd(self.dz, None, self.xs, wi, self.group_offsets,
                                          self.dxs, self.dwi, self.status, self.ws, d, stream)
        B.moe_permute_bwd(self.dxs, self.pos, self.dx, d, stream)
        return self.dx
