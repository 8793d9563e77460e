"""FP8 MLP blocks and stacks over the C ABI (marshalling only).

One block is fc1 (d -> ffn) -> GELU -> fc2 (ffn -> d), both linears FP8
("Native FP8 MLP reconstruction": FP8 only in the MLP linears, micro 64 x
2048 tokens with gradient accumulation over 4 microbatches).  A stack chains
blocks; gradient accumulation sums each weight's bf16 dW into an fp32
accumulator in microbatch order.  Weights go through the library's weight
cache: with use_cache the FP8 copies are made on the first microbatch of a
cycle and reused (is_first_microbatch True/False); without it every
microbatch re-quantizes (is_first_microbatch None).
"""
from __future__ import annotations

import torch

import fp8_mixed_precision_gb300 as fp
from fp8_mixed_precision_gb300 import synthetic as syn


class FP8MLPStack:
    """fused (block recipe only): GELU forward is fused with the quantization
    of fc2's input and GELU backward with the quantization of fc1's incoming
    gradient, so the bf16 A and dH tensors are never written; results are
    bitwise identical to the unfused path."""

    def __init__(self, d: int, ffn: int, n_layers: int, n_tokens: int, recipe: str = "block",
                 device="cuda", seed: int = 43, fused: bool = False):
        self.d, self.ffn, self.L, self.N, self.recipe = d, ffn, n_layers, n_tokens, recipe
        self.fused = bool(fused) and recipe == "block"
        dev = torch.device(device)
        self.dev = dev
        self.cache = fp.WeightCache()
        self.w1, self.w2, self.h1, self.h2 = [], [], [], []
        for l in range(n_layers):
            w1 = syn.bf16_normal((ffn, d), 0.02, seed + 2 * l, device=dev)
            w2 = syn.bf16_normal((d, ffn), 0.02, seed + 2 * l + 1, device=dev)
            self.w1.append(w1)
            self.w2.append(w2)
            self.h1.append(self.cache.register(w1, recipe))
            self.h2.append(self.cache.register(w2, recipe))
        self.dw1 = [torch.zeros((ffn, d), dtype=torch.float32, device=dev) for _ in range(n_layers)]
        self.dw2 = [torch.zeros((d, ffn), dtype=torch.float32, device=dev) for _ in range(n_layers)]
        N = n_tokens
        # one workspace serves every linear (they run in order on one stream)
        self.ws = max(fp.linear_workspace(recipe, N, d, ffn, dev),
                      fp.linear_workspace(recipe, N, ffn, d, dev), key=lambda t: t.numel())
        # per-layer saved state: fc1 context, pre-GELU H, GELU output A, fc2 context
        self.ctx1 = [fp.LinearContext(fp._empty_bytes(fp._ctx_bytes(recipe, N, d), dev), N, d)
                     for _ in range(n_layers)]
        self.ctx2 = [fp.LinearContext(fp._empty_bytes(fp._ctx_bytes(recipe, N, ffn), dev), N, ffn)
                     for _ in range(n_layers)]
        self.H = [torch.empty((N, ffn), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
        if self.fused:
            # fc2's quantized input: rowwise in a buffer, transposed inside fc2's context
            self.Aq = [fp.QuantizedTensor(N, ffn, "act", dev,
                                          col_ptrs=fp.fp8_linear_ctx_layout(recipe, self.ctx2[l]))
                       for l in range(n_layers)]
            self.dHq = fp.QuantizedTensor(N, ffn, "grad", dev)
            self.A = None
        else:
            self.A = [torch.empty((N, ffn), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
        self.Y = [torch.empty((N, d), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
        self.dA = torch.empty((N, ffn), dtype=torch.bfloat16, device=dev)
        self.dH = None if self.fused else torch.empty((N, ffn), dtype=torch.bfloat16, device=dev)
        self.g = [torch.empty((N, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.dwb1 = torch.empty((ffn, d), dtype=torch.bfloat16, device=dev)
        self.dwb2 = torch.empty((d, ffn), dtype=torch.bfloat16, device=dev)
        self.version = 0
        self.requantized = 0

    def zero_grad(self):
        for t in self.dw1 + self.dw2:
            t.zero_()

    def microbatch(self, x: torch.Tensor, dy: torch.Tensor, use_cache: bool):
        """Forward and backward of one microbatch; returns (Y of the last
        layer, dX of the first layer).  dW accumulate into self.dw1/dw2."""
        r, c = self.recipe, self.cache
        h = x
        for l in range(self.L):
            self.requantized += c.get(self.h1[l], self.version, use_cache)
            fp.fp8_linear_fwd(h, c, self.h1[l], r, ws=self.ws, y=self.H[l], ctx=self.ctx1[l])
            self.requantized += c.get(self.h2[l], self.version, use_cache)
            if self.fused:
                fp.fp8_gelu_quantize(self.H[l], self.Aq[l], r)
                fp.fp8_linear_fwd_quantized(self.Aq[l], c, self.h2[l], r, self.ws, self.Y[l])
            else:
                fp.fp8_gelu_fwd(self.H[l], out=self.A[l])
                fp.fp8_linear_fwd(self.A[l], c, self.h2[l], r, ws=self.ws, y=self.Y[l],
                                  ctx=self.ctx2[l])
            h = self.Y[l]
        g = dy
        for l in reversed(range(self.L)):
            fp.fp8_linear_bwd(g, self.ctx2[l], c, self.h2[l], r, ws=self.ws, dx=self.dA,
                              dw=self.dwb2)
            fp.fp8_grad_accumulate(self.dw2[l], self.dwb2)
            out = self.g[l % 2]
            if self.fused:
                fp.fp8_gelu_bwd_quantize(self.dA, self.H[l], self.dHq, r)
                fp.fp8_linear_bwd_quantized(self.dHq, self.ctx1[l], c, self.h1[l], r, self.ws, out,
                                            self.dwb1)
            else:
                fp.fp8_gelu_bwd(self.dA, self.H[l], out=self.dH)
                fp.fp8_linear_bwd(self.dH, self.ctx1[l], c, self.h1[l], r, ws=self.ws, dx=out,
                                  dw=self.dwb1)
            fp.fp8_grad_accumulate(self.dw1[l], self.dwb1)
            g = out
        return self.Y[self.L - 1], g

    def step(self, xs, dys, use_cache: bool, keep_outputs: bool = True):
        """One gradient-accumulation cycle over the microbatches (weights are
        unchanged within it).  Returns the per-microbatch (Y, dX) pairs,
        copied out of the internal buffers when keep_outputs."""
        self.cache.begin_cycle()
        self.version += 1
        self.zero_grad()
        outs = []
        for x, dy in zip(xs, dys):
            y, dx = self.microbatch(x, dy, use_cache)
            if keep_outputs:
                outs.append((y.clone(), dx.clone()))
        return outs
