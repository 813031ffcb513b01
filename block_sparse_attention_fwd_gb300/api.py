"""User-facing BackLite attention on the bl_attn C ABI.

``BLAttention(negl_prob)`` mirrors the module the "BackLite" README describes
(Usage, Forward signature): it is called as
``attn(query, key, value, scale=None, return_softmax_lse=False, tile_stats=None)``
on (batch, seq_len, heads, head_dim) bf16 tensors, with key/value carrying
``heads_k`` heads.  With negl_prob > 0 the forward records tile statistics
(allocating the buffer unless one is passed, README, Note) and the backward
builds the block-sparse mask from them before running the sparse backward
(How It Works, Phase 2).  With no statistics buffer passed, the forward
keeps only the tile weights d_ij the mask reads (the "Introducing BackLite"
post, Using Sparsity), reduced in its epilogue.  negl_prob = 0 records nothing and runs the dense
backward (Key properties).  ``BL_VERBOSE=1`` prints mask density per head
after each mask pass (README, Debugging, names the same kind of switch).
``causal=True`` (optionally with ``window=W``) gives decoder attention, with
the sliding windows of the "Introducing BackLite" post's Nanochat runs
(Training Nanochat).  ``BLAttention.varlen(q, k, v, cu_seqlens)`` runs the
same chain on a packed variable-length batch ([total, heads, head_dim]
tensors, host offsets cu_seqlens), each sequence attending only to itself.

PyTorch only allocates memory and supplies the stream; all arithmetic runs in
libbl_attn.so.
"""
from __future__ import annotations

import math
import os

import torch

from . import _lib


def default_tiles(n: int, d: int):
    """Tile sizes used when the caller does not choose: 128 x 128."""
    return 128, 128


class _BLAttnFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, negl_prob, block_q, block_k, tile_stats, causal, window):
        B, n, H, d = q.shape
        Hk = k.shape[2]
        shape = _lib.make_shape(B, n, H, Hk, d, block_q, block_k, causal, window)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
        stats = logw = None
        if negl_prob > 0:
            T_r, T_c = _lib.tiles(shape)
            if tile_stats is None and _lib.fwd_tile_weights_supported(shape):
                # Only the T_r x T_c tile weights outlive the forward; the
                # statistics rows stay in a scratch freed on return.
                logw = torch.empty((B, H, T_r, T_c), dtype=torch.float32, device=q.device)
                ws = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8,
                                 device=q.device)
                _lib.attn_fwd_tile_weights(shape, q, k, v, scale, o, lse, logw, workspace=ws)
            else:
                want = (B, H, T_c, T_r * block_q)
                stats = tile_stats if tile_stats is not None else torch.empty(
                    want, dtype=torch.float32, device=q.device)
        if logw is None:
            _lib.attn_fwd(shape, q, k, v, scale, o, lse, stats)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.stats, ctx.logw = stats, logw
        ctx.cfg = (shape, scale, negl_prob)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, g_o, _g_lse):
        q, k, v, o, lse = ctx.saved_tensors
        shape, scale, negl_prob = ctx.cfg
        g_o = g_o.contiguous()
        lists = None
        if ctx.stats is not None or ctx.logw is not None:
            lists = _lib.alloc_lists(shape, q.device)
            if ctx.logw is not None:
                _lib.mask_from_tile_weights(shape, ctx.logw, negl_prob, lists)
            else:
                _lib.mask_from_stats(shape, ctx.stats, lse, negl_prob, lists)
            if os.environ.get("BL_VERBOSE") == "1":
                m = lists["mask"].float()
                dens = m.mean(dim=(2, 3)).cpu()
                print(f"[bl_attn] mask density per (batch, head): {dens.tolist()} "
                      f"backward skip fraction {1.0 - float(m.mean()):.4f}")
        g_q = torch.empty_like(q)
        g_k = torch.empty_like(k)
        g_v = torch.empty_like(v)
        ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=q.device)
        _lib.attn_bwd(shape, q, k, v, o, g_o, lse, scale, lists, g_q, g_k, g_v, ws)
        return g_q, g_k, g_v, None, None, None, None, None, None, None


class _BLAttnVarlenFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, vl, scale, negl_prob):
        o = torch.empty_like(q)
        lse = torch.empty(vl.sizes["lse"], dtype=torch.float32, device=q.device)
        stats = logw = None
        if negl_prob > 0 and _lib.fwd_tile_weights_supported_varlen(vl):
            logw = torch.empty(vl.sizes["mask"], dtype=torch.float32, device=q.device)
            ws = torch.empty(_lib.fwd_workspace_bytes_varlen(vl), dtype=torch.uint8,
                             device=q.device)
            _lib.attn_fwd_tile_weights_varlen(vl, q, k, v, scale, o, lse, logw, workspace=ws)
        else:
            if negl_prob > 0:
                stats = torch.empty(vl.sizes["tile_stats"], dtype=torch.float32,
                                    device=q.device)
            _lib.attn_fwd_varlen(vl, q, k, v, scale, o, lse, stats)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.stats, ctx.logw = stats, logw
        ctx.cfg = (vl, scale, negl_prob)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, g_o, _g_lse):
        q, k, v, o, lse = ctx.saved_tensors
        vl, scale, negl_prob = ctx.cfg
        lists = None
        if ctx.stats is not None or ctx.logw is not None:
            lists = _lib.alloc_varlen_lists(vl, q.device)
            if ctx.logw is not None:
                _lib.mask_from_tile_weights_varlen(vl, ctx.logw, negl_prob, lists)
            else:
                _lib.mask_from_stats_varlen(vl, ctx.stats, lse, negl_prob, lists)
        g_q, g_k, g_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device=q.device)
        _lib.attn_bwd_varlen(vl, q, k, v, o, g_o.contiguous(), lse, scale, lists, g_q, g_k, g_v,
                             ws)
        return g_q, g_k, g_v, None, None, None


class BLAttention(torch.nn.Module):
    """Attention whose backward skips the lightest tiles (negl_prob of the mass)."""

    def __init__(self, negl_prob: float = 0.05, block_q: int | None = None,
                 block_k: int | None = None, causal: bool = False, window: int = 0):
        super().__init__()
        if not (0.0 <= negl_prob < 1.0):
            raise ValueError("negl_prob must lie in [0, 1)")
        if window < 0 or (window and not causal):
            raise ValueError("a sliding window needs causal=True")
        self.negl_prob = float(negl_prob)
        self.block_q, self.block_k = block_q, block_k
        self.causal, self.window = bool(causal), int(window)

    def forward(self, query, key, value, scale=None, return_softmax_lse=False, tile_stats=None):
        d = query.shape[-1]
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        bq, bk = default_tiles(query.shape[1], d)
        bq = self.block_q or bq
        bk = self.block_k or bk
        q, k, v = (t.contiguous() for t in (query, key, value))
        o, lse = _BLAttnFn.apply(q, k, v, float(scale), self.negl_prob, bq, bk, tile_stats,
                                 int(self.causal), self.window)
        return (o, lse) if return_softmax_lse else o

    def varlen(self, query, key, value, cu_seqlens, scale=None, return_softmax_lse=False):
        """The same attention on a packed batch: query [total, H, d], key/value
        [total, Hk, d], cu_seqlens the nseq + 1 token offsets (a host sequence
        or CPU tensor).  Returns O [total, H, d] and, if asked, the flat LSE
        (per sequence a [H, n_s] block at offset H * cu_seqlens[s])."""
        total, H, d = query.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        bq, bk = default_tiles(total, d)
        vl = _lib.Varlen(cu_seqlens, H, key.shape[1], d, self.block_q or bq, self.block_k or bk,
                         int(self.causal), self.window)
        if vl.total != total:
            raise ValueError(f"cu_seqlens covers {vl.total} tokens, query has {total}")
        q, k, v = (t.contiguous() for t in (query, key, value))
        o, lse = _BLAttnVarlenFn.apply(q, k, v, vl, float(scale), self.negl_prob)
        return (o, lse) if return_softmax_lse else o
