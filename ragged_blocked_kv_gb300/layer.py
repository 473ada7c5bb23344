"""A decoder layer around the library's attention pass, every step a library
kernel (tensor-core GEMMs with fused epilogues, RMSNorm, the KV append and
ragged attention).

DeepSpeed-FastGen paper summary page, idea I1: a pass's latency follows its
token count; the layer's projections are that token-proportional work.  The
layer is a Llama-2-7B decoder layer (pre-RMSNorm, QKV and output projections,
SwiGLU MLP, residuals; rotary embeddings left out), random bf16 weights.

Weights as stored here: ``w_qkv`` [(H_q + 2 H_kv) D][hidden] (Q rows, then K,
then V), ``w_o`` [hidden][H_q D], ``w_gu`` [2 ffn][hidden] with the gate and
up rows interleaved in blocks of 128 (rows 256 b .. 256 b + 127 are gate rows
128 b .. 128 b + 127, the next 128 the up rows of the same outputs: the GEMM's
SwiGLU epilogue pairs them), ``w_down`` [hidden][ffn], ``g_attn`` and
``g_mlp`` [hidden].
"""
from __future__ import annotations

import math
from typing import Dict, Optional


def interleave_gate_up(w_gate, w_up):
    """[ffn][hidden] gate and up weights -> the [2 ffn][hidden] block layout of
    the SwiGLU epilogue (ffn a multiple of 128)."""
    import torch
    ffn, hidden = w_gate.shape
    if ffn % 128:
        raise ValueError("ffn must be a multiple of 128")
    g = w_gate.reshape(ffn // 128, 128, hidden)
    u = w_up.reshape(ffn // 128, 128, hidden)
    return torch.stack([g, u], dim=1).reshape(2 * ffn, hidden).contiguous()


def random_weights(hidden: int, num_heads_q: int, num_heads_kv: int, head_dim: int, ffn: int,
                   seed: int, device: str = "cuda") -> Dict[str, "object"]:
    """Seeded random bf16 weights: N(0,1) / sqrt(fan_in); norm weights 1 +
    N(0,1) / 10.  Gate and up are returned separately (``w_gate``, ``w_up``)
    and interleaved (``w_gu``)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    def w(out_f, in_f):
        return (torch.randn(out_f, in_f, generator=gen, device=device) /
                math.sqrt(in_f)).to(torch.bfloat16)

    nq, nkv = num_heads_q * head_dim, num_heads_kv * head_dim
    ws = {
        "w_qkv": w(nq + 2 * nkv, hidden),
        "w_o": w(hidden, nq),
        "w_gate": w(ffn, hidden),
        "w_up": w(ffn, hidden),
        "w_down": w(hidden, ffn),
        "g_attn": (1.0 + torch.randn(hidden, generator=gen, device=device) / 10).to(torch.bfloat16),
        "g_mlp": (1.0 + torch.randn(hidden, generator=gen, device=device) / 10).to(torch.bfloat16),
    }
    ws = {k: v.contiguous() for k, v in ws.items()}
    ws["w_gu"] = interleave_gate_up(ws["w_gate"], ws["w_up"])
    return ws


class DecoderLayer:
    """One layer's weights and its forward pass over a composed pass."""

    def __init__(self, rbkv, weights: dict, num_heads_q: int, num_heads_kv: int, head_dim: int,
                 eps: float = 1e-5):
        self.rbkv = rbkv
        self.w = weights
        self.hq, self.hkv, self.d = num_heads_q, num_heads_kv, head_dim
        self.eps = eps

    def buffers(self, max_tokens: int, device: str = "cuda") -> dict:
        """Fixed activation buffers of max_tokens rows (for forward_into)."""
        import torch
        hidden = self.w["w_o"].shape[0]
        ffn = self.w["w_down"].shape[1]
        bf = dict(dtype=torch.bfloat16, device=device)
        return {"a": torch.empty(max_tokens, hidden, **bf),
                "q": torch.empty(max_tokens, self.hq, self.d, **bf),
                "k": torch.empty(max_tokens, self.hkv, self.d, **bf),
                "v": torch.empty(max_tokens, self.hkv, self.d, **bf),
                "o": torch.empty(max_tokens, self.hq, self.d, **bf),
                "h": torch.empty(max_tokens, hidden, **bf),
                "b": torch.empty(max_tokens, hidden, **bf),
                "act": torch.empty(max_tokens, ffn, **bf),
                "gemm_ws": torch.empty(max(256, self.gemm_workspace_bytes(max_tokens)),
                                       dtype=torch.uint8, device=device)}

    def gemm_workspace_bytes(self, rows: int) -> int:
        """Split-K workspace enough for every projection of up to `rows` rows
        (each product splits less as rows grow; every row count is tried up
        to one tile)."""
        w = self.w
        shapes = [w["w_qkv"].shape, w["w_o"].shape, w["w_gu"].shape, w["w_down"].shape]
        need = 0
        for r in sorted({min(rows, x) for x in (1, 128, 256, 512, 1024, 2048, rows)}):
            for n, k in shapes:
                need = max(need, self.rbkv.gemm_workspace_bytes(r, n, k))
        return need

    def forward_into(self, x, out, buf: dict, attend, rows: int, stream=None) -> None:
        """The layer on the first `rows` rows of fixed buffers: x -> out, with
        attend(q, k, v, o) running the KV append and attention (a plain pass
        or a frame); allocates nothing, so it can be captured in a graph."""
        rb, w = self.rbkv, self.w
        T = rows
        a, h, b, act = buf["a"][:T], buf["h"][:T], buf["b"][:T], buf["act"][:T]
        q, k, v, o = buf["q"][:T], buf["k"][:T], buf["v"][:T], buf["o"][:T]
        rb.rmsnorm(x, w["g_attn"], y=a, eps=self.eps, stream=stream)
        ws = buf["gemm_ws"]
        rb.gemm_qkv(a, w["w_qkv"], self.hq, self.hkv, self.d, out=(q, k, v), workspace=ws,
                    stream=stream)
        attend(q, k, v, o)
        rb.gemm(o.view(T, self.hq * self.d), w["w_o"], c=h, residual=x, epilogue="residual",
                workspace=ws, stream=stream)
        rb.rmsnorm(h, w["g_mlp"], y=b, eps=self.eps, stream=stream)
        rb.gemm(b, w["w_gu"], c=act, epilogue="swiglu", workspace=ws, stream=stream)
        rb.gemm(act, w["w_down"], c=out, residual=h, epilogue="residual", workspace=ws,
                stream=stream)

    def forward(self, p, x, k_cache, v_cache, workspace=None, stream=None,
                status=None) -> dict:
        """x: [T][hidden] bf16 for the pass's rows; appends the pass's K and V
        to the caches and returns the layer's output and intermediates."""
        rb, w = self.rbkv, self.w
        T, hidden = x.shape
        a = rb.rmsnorm(x, w["g_attn"], eps=self.eps, stream=stream)
        q, k, v = rb.gemm_qkv(a, w["w_qkv"], self.hq, self.hkv, self.d, status=status,
                              stream=stream)
        rb.kv_append(p, k, v, k_cache, v_cache, stream=stream)
        o = rb.ragged_attention(p, q, k_cache, v_cache, workspace=workspace, stream=stream)
        h = rb.gemm(o.view(T, self.hq * self.d), w["w_o"], residual=x, epilogue="residual",
                    status=status, stream=stream)
        b = rb.rmsnorm(h, w["g_mlp"], eps=self.eps, stream=stream)
        act = rb.gemm(b, w["w_gu"], epilogue="swiglu", status=status, stream=stream)
        out = rb.gemm(act, w["w_down"], residual=h, epilogue="residual", status=status,
                      stream=stream)
        return {"a": a, "q": q, "k": k, "v": v, "o": o, "h": h, "b": b, "act": act, "out": out}
