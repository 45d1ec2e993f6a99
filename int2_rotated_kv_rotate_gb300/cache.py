"""A torch-facing handle on one cache of the C library (marshalling only).

torch allocates the device block and the decode workspace; every operation is one call
of the C ABI (see include/oscar.h for semantics and layouts).
"""
from __future__ import annotations

import torch

from . import _native as N


class KVCache:
    """One cache: INT2 mixed-precision (fmt=N.OSCAR_FORMAT_INT2, or N.OSCAR_FORMAT_INT2_CM with
    channel-major value pages) or plain BF16 pages (N.OSCAR_FORMAT_BF16)."""

    def __init__(self, *, fmt: int = N.OSCAR_FORMAT_INT2, n_q_heads: int, n_kv_heads: int, group: int = 128,
                 n_sink: int = 4, window: int = 128, n_layers: int = 1, max_requests: int = 1, max_pages: int,
                 max_pages_per_request: int, head_dim: int = 128, device="cuda"):
        self.cfg = N.oscar_config(fmt, head_dim, n_q_heads, n_kv_heads, group, 64, n_sink, window, n_layers,
                                  max_requests, max_pages, max_pages_per_request)
        self.nbytes = N.oscar_cache_device_bytes(self.cfg)
        self.device = torch.device(device)
        self.mem = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        self.handle = N.oscar_cache_create(self.cfg, self.mem, self.nbytes)
        self.layout = N.oscar_cache_layout(self.handle)
        self.workspace = None
        self.fmt = fmt
        self.is_int2 = fmt in (N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM)
        self._rows = None  # rows of k_new / v_new the pending reservation expects
        self._n_plan = None  # requests of the current decode plan

    # ------------------------------------------------------------------ lifecycle
    def close(self) -> None:
        if getattr(self, "handle", None):
            N.oscar_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ params / requests
    def set_layer_params(self, layer: int, R_K, R_V, clip_K, clip_V, stream=None) -> None:
        f = lambda t: torch.as_tensor(t, dtype=torch.float32).contiguous().cpu()  # noqa: E731
        N.oscar_set_layer_params(self.handle, layer, f(R_K), f(R_V), f(clip_K), f(clip_V), stream)

    def stats(self):
        """(free pages, free request slots)."""
        return N.oscar_cache_stats(self.handle)

    def alloc(self) -> int:
        return N.oscar_request_alloc(self.handle)

    def free(self, slot: int) -> None:
        N.oscar_request_free(self.handle, slot)

    def info(self, slot: int):
        return N.oscar_request_info(self.handle, slot)

    def pages(self, slot: int):
        return N.oscar_request_pages(self.handle, slot, self.info(slot)[2])

    def share_prefix(self, dst: int, src: int, n_tokens: int, stream=None) -> None:
        N.oscar_request_share_prefix(self.handle, dst, src, n_tokens, stream)

    # ------------------------------------------------------------------ append
    def reserve(self, slots, n_new, stream=None) -> None:
        N.oscar_reserve(self.handle, slots, n_new, stream)
        self._rows = int(sum(int(n) for n in n_new))

    def _check_tokens(self, k_new, v_new) -> None:
        shape = (self._rows, self.cfg.n_kv_heads, self.cfg.head_dim)
        for t in (k_new, v_new):
            if (tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_contiguous()
                    or t.device != self.mem.device):
                raise ValueError(f"token tensors must be contiguous bf16 {shape} on {self.mem.device}")

    def quantize_append(self, layer: int, k_new, v_new, stream=None) -> None:
        self._check_tokens(k_new, v_new)
        N.oscar_quantize_append(self.handle, layer, k_new, v_new, stream)

    def bf16_append(self, layer: int, k_new, v_new, stream=None) -> None:
        self._check_tokens(k_new, v_new)
        N.oscar_bf16_append(self.handle, layer, k_new, v_new, stream)

    def append(self, layer: int, k_new, v_new, stream=None) -> None:
        if self.is_int2:
            self.quantize_append(layer, k_new, v_new, stream)
        else:
            self.bf16_append(layer, k_new, v_new, stream)

    def commit(self) -> None:
        N.oscar_commit_append(self.handle)
        self._rows = None
        self._n_plan = None

    # ------------------------------------------------------------------ decode
    def plan(self, slots, max_split_pages: int = 0, stream=None, flags: int = 0) -> int:
        N.oscar_plan_decode_ex(self.handle, slots, max_split_pages, flags, stream)
        self._n_plan = len(list(slots))
        need = N.oscar_decode_workspace_bytes(self.handle)
        if self.workspace is None or self.workspace.numel() < need:
            # sized for every plan of the cache, once: launches captured into a graph keep
            # this pointer across later plans
            full = N.oscar_decode_workspace_max_bytes(self.handle)
            self.workspace = torch.empty(max(need, full, 256), dtype=torch.uint8, device=self.device)
        return need

    def plan_info(self):
        return N.oscar_plan_info(self.handle)

    def _check_decode(self, q, out, out_f32):
        shape = (self._n_plan, self.cfg.n_q_heads, self.cfg.head_dim)
        if tuple(q.shape) != shape or q.dtype != torch.bfloat16 or not q.is_contiguous() or q.device != self.mem.device:
            raise ValueError(f"q must be contiguous bf16 {shape} on {self.mem.device}")
        if out is None:
            out = torch.empty_like(q)
        if tuple(out.shape) != shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
            raise ValueError("out must be contiguous bf16 like q")
        if out_f32 is not None and (tuple(out_f32.shape) != shape or out_f32.dtype != torch.float32
                                    or not out_f32.is_contiguous()):
            raise ValueError("out_f32 must be contiguous fp32 like q")
        return out

    def decode(self, layer: int, q, out=None, out_f32=None, stream=None):
        out = self._check_decode(q, out, out_f32)
        if self.is_int2:
            N.oscar_decode_attention(self.handle, layer, q, out, self.workspace, out_f32, stream)
        else:
            N.oscar_bf16_decode_attention(self.handle, layer, q, out, self.workspace, out_f32, stream)
        return out

    def append_decode(self, layer: int, k_new, v_new, q, out=None, out_f32=None, stream=None):
        """quantize_append then decode of `layer` in one launch (INT2 format; plan made
        during the reservation over every reserved slot)."""
        self._check_tokens(k_new, v_new)
        out = self._check_decode(q, out, out_f32)
        N.oscar_append_decode_attention(self.handle, layer, k_new, v_new, q, out, self.workspace, out_f32, stream)
        return out

    def status(self, stream=None):
        return N.oscar_get_status(self.handle, stream)

    # ------------------------------------------------------------------ raw reads (tests)
    def _bytes(self, offset: int, n: int) -> torch.Tensor:
        return self.mem[offset:offset + n]

    def int2_rows(self, layer: int, slot: int, kvh: int, kv: int, positions):
        """Device-stored 32-byte code rows and scale/zero words of INT2 positions (host)."""
        H = self.cfg.n_kv_heads
        ng = 128 // self.cfg.group
        pos = torch.as_tensor(list(positions) if not torch.is_tensor(positions) else positions, dtype=torch.long)
        if pos.numel() == 0:
            return torch.empty((0, 32), dtype=torch.uint8), torch.empty((0, ng * 2), dtype=torch.int16)
        pages = torch.tensor(self.pages(slot), dtype=torch.long)
        phys = pages[pos // 64]
        t = pos % 64
        code_head = self.layout.codes_page_bytes
        sz_head = self.layout.sz_page_bytes
        code_layer = self.cfg.max_pages * H * code_head
        sz_layer = self.cfg.max_pages * H * sz_head
        c0 = self.layout.codes + layer * code_layer + (phys * H + kvh) * code_head + kv * 64 * 32 + t * 32
        s0 = self.layout.sz + layer * sz_layer + (phys * H + kvh) * sz_head + kv * 64 * ng * 4 + t * ng * 4
        dev = self.mem.device
        is_ = (s0[:, None] + torch.arange(ng * 4)[None, :]).to(dev)
        sz = self.mem[is_].cpu().contiguous().view(torch.int16)
        if self.fmt == N.OSCAR_FORMAT_INT2_CM and kv == 1:
            return self._cm_rows(c0 - t * 32, t), sz
        ic = (c0[:, None] + torch.arange(32)[None, :]).to(dev)
        rows = self.mem[ic].cpu()
        return rows, sz

    def _cm_rows(self, vblock: torch.Tensor, t: torch.Tensor) -> torch.Tensor:
        """Token-major 32-byte rows of positions t (in their pages) rebuilt from channel-major
        value blocks at byte offsets vblock: word 128 b + c holds channel c of tokens
        16 b .. 16 b + 15, token 16 b + 8 h + f at bit 16 h + 2 f."""
        dev = self.mem.device
        c = torch.arange(128)
        word0 = vblock + 4 * (128 * (t // 16))
        iw = (word0[:, None, None] + 4 * c[None, :, None] + torch.arange(4)[None, None, :]).to(dev)
        words = self.mem[iw].cpu().to(torch.int64)
        words = words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24)  # [n, 128]
        sh = (16 * ((t // 8) % 2) + 2 * (t % 8))[:, None]
        codes = (words >> sh) & 3  # [n, 128] code of channel c
        f, w, h = c // 16, (c % 16) // 2, c % 2  # channel c = 16 f + 2 w + h: bit 32 w + 16 h + 2 f of the row
        row_words = torch.zeros((t.numel(), 8), dtype=torch.int64)
        row_words.scatter_add_(1, w[None, :].expand(t.numel(), 128), codes << (16 * h + 2 * f)[None, :])
        row_words = torch.where(row_words >= 2**31, row_words - 2**32, row_words)  # two's complement words
        return row_words.to(torch.int32).view(torch.uint8).reshape(t.numel(), 32)

    def _head_block(self, pool_off: int, per_head: int, slot: int, layer: int, kvh: int):
        H = self.cfg.n_kv_heads
        off = pool_off + ((slot * self.cfg.n_layers + layer) * H + kvh) * per_head
        return self.mem[off:off + per_head]

    def sink_tokens(self, layer: int, slot: int, kvh: int, kv: int) -> torch.Tensor:
        S = self.cfg.n_sink
        blk = self._head_block(self.layout.sink, self.layout.sink_bytes_per_head, slot, layer, kvh)
        return blk.view(torch.int16).view(2, S, 128)[kv].cpu()

    def ring_tokens(self, layer: int, slot: int, kvh: int, kv: int) -> torch.Tensor:
        W = self.cfg.window
        blk = self._head_block(self.layout.ring, self.layout.ring_bytes_per_head, slot, layer, kvh)
        return blk.view(torch.int16).view(2, W, 128)[kv].cpu()
