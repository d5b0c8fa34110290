"""Python binding of libpkv, the paged-KV decode step for GB300 (sm_103a).

The functions here have the names of the C ABI in ``include/pkv.h`` and do
argument marshalling only: they check dtypes, devices and contiguity of torch
tensors and pass their data pointers (and the current CUDA stream) to the
library.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback.  If ``libpkv.so`` has not been built, importing the
binding's functions raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_EINVAL, PKV_ERANGE, PKV_ENOMEM, PKV_ECUDA, PKV_EWORKSPACE, PKV_EDEVICE, PKV_ENOTIMPL = \
    0, -1, -2, -3, -4, -5, -6, -7
PKV_DEVERR_POSITION, PKV_DEVERR_PAGE, PKV_DEVERR_ROW, PKV_DEVERR_SLOT, PKV_DEVERR_TIMEOUT = 1, 2, 4, 8, 16

# Every symbol include/pkv.h declares.
ABI_SYMBOLS = ("pkv_config_default", "pkv_strerror", "pkv_pool_alloc", "pkv_pool_wrap", "pkv_pool_free",
               "pkv_pool_kv", "pkv_workspace_bytes", "pkv_decode", "pkv_step", "pkv_prefill", "pkv_check_errors",
               "pkv_set_ctas", "pkv_set_wait_limit", "pkv_timer_enable", "pkv_timer_read", "pkv_decode_static",
               "pkv_linear_workspace_bytes", "pkv_linear", "pkv_qkv_proj", "pkv_qkv_proj_append",
               "pkv_decode_appended", "pkv_output_gate")

# Size of the scratch array pkv_decode_static uses in place of a workspace.
PKV_STATIC_SCRATCH_BYTES = 32 << 20


class PkvConfig(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_seq", ctypes.c_int),
                ("rope_theta", ctypes.c_double), ("eps", ctypes.c_double), ("rotary_dim", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {pkv_strerror(code)} ({code})")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpkv.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libpkv.so not found at {path}: build it first (python -c 'import __graft_entry__ as g; "
                           f"g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(PkvConfig)
    sig = {
        "pkv_config_default": ([cfgp], i32),
        "pkv_strerror": ([i32], ctypes.c_char_p),
        "pkv_pool_alloc": ([cfgp, i32, vp, ctypes.POINTER(vp)], i32),
        "pkv_pool_wrap": ([cfgp, i32, vp, vp, vp, ctypes.POINTER(vp)], i32),
        "pkv_pool_free": ([vp], i32),
        "pkv_pool_kv": ([vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64)], i32),
        "pkv_workspace_bytes": ([vp, i32, i32, i32, ctypes.POINTER(sz)], i32),
        "pkv_decode": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp], i32),
        "pkv_step": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, sz, vp], i32),
        "pkv_prefill": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, sz, vp], i32),
        "pkv_check_errors": ([vp, vp, ctypes.POINTER(ctypes.c_uint32)], i32),
        "pkv_set_ctas": ([vp, i32], i32),
        "pkv_set_wait_limit": ([vp, i64], i32),
        "pkv_timer_enable": ([vp, i32], i32),
        "pkv_timer_read": ([vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)], i32),
        "pkv_decode_static": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp], i32),
        "pkv_linear_workspace_bytes": ([vp, i32, i32, i32, ctypes.POINTER(sz)], i32),
        "pkv_linear": ([vp, vp, vp, vp, i32, i32, i32, vp, sz, vp], i32),
        "pkv_qkv_proj": ([vp, vp, vp, i32, i32, vp, vp, vp, vp], i32),
        "pkv_qkv_proj_append": ([vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, vp, vp], i32),
        "pkv_decode_appended": ([vp, vp, vp, vp, i32, i32, vp, vp, sz, vp], i32),
        "pkv_output_gate": ([vp, vp, vp, i32, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != PKV_OK:
        raise PkvError(rc, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor | None, dtype: torch.dtype, what: str, allow_none: bool = False) -> ctypes.c_void_p:
    if t is None:
        if allow_none:
            return ctypes.c_void_p(None)
        raise ValueError(f"{what} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------ C ABI, one function each

def pkv_strerror(code: int) -> str:
    return load_library().pkv_strerror(int(code)).decode()


def pkv_config_default() -> PkvConfig:
    c = PkvConfig()
    _check(load_library().pkv_config_default(ctypes.byref(c)), "pkv_config_default")
    return c


def _cfg(cfg) -> PkvConfig:
    if cfg is None:
        return pkv_config_default()
    if isinstance(cfg, PkvConfig):
        return cfg
    c = pkv_config_default()
    for k, v in dict(cfg).items():
        setattr(c, k, v)
    return c


def pkv_pool_alloc(cfg, num_pages: int, stream=None) -> ctypes.c_void_p:
    out = ctypes.c_void_p()
    _check(load_library().pkv_pool_alloc(ctypes.byref(_cfg(cfg)), int(num_pages), _stream(stream),
                                         ctypes.byref(out)), "pkv_pool_alloc")
    return out


def pkv_pool_wrap(cfg, num_pages: int, k: torch.Tensor, v: torch.Tensor, stream=None) -> ctypes.c_void_p:
    out = ctypes.c_void_p()
    _check(load_library().pkv_pool_wrap(ctypes.byref(_cfg(cfg)), int(num_pages), _dev(k, torch.bfloat16, "k"),
                                        _dev(v, torch.bfloat16, "v"), _stream(stream), ctypes.byref(out)),
           "pkv_pool_wrap")
    return out


def pkv_pool_free(pool) -> None:
    _check(load_library().pkv_pool_free(pool), "pkv_pool_free")


def pkv_pool_kv(pool):
    k, v, n = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int64()
    _check(load_library().pkv_pool_kv(pool, ctypes.byref(k), ctypes.byref(v), ctypes.byref(n)), "pkv_pool_kv")
    return k.value, v.value, n.value


def pkv_workspace_bytes(pool, rows: int, pages: int, prefill_tokens: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(load_library().pkv_workspace_bytes(pool, int(rows), int(pages), int(prefill_tokens), ctypes.byref(n)),
           "pkv_workspace_bytes")
    return n.value


def _table(table, rows, pages):
    """(pointer, rows, pages) of a page table, or of the contiguous-row layout when ``table`` is None."""
    if table is None:
        if rows is None or pages is None:
            raise ValueError("without a table, rows and pages are required")
        return ctypes.c_void_p(None), int(rows), int(pages)
    if table.dim() != 2:
        raise ValueError(f"table must be [rows][pages], got {tuple(table.shape)}")
    return _dev(table, torch.int32, "table"), int(table.shape[0]), int(table.shape[1])


def pkv_decode(pool, q, k, v, q_norm_w, k_norm_w, positions, table, out, workspace, stream=None,
               pages=None) -> None:
    """decode_paged; ``table=None`` with ``pages`` is decode_rows over contiguous rows."""
    tp, rows, pages = _table(table, positions.shape[0], pages)
    _check(load_library().pkv_decode(
        pool, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(q_norm_w, torch.bfloat16, "q_norm_w"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(positions, torch.int32, "positions"), tp, rows, pages,
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)), "pkv_decode")


def pkv_decode_static(pool, q, k, v, q_norm_w, k_norm_w, positions, table, out, stream=None, pages=None) -> None:
    """pkv_decode without a workspace: the library's static scratch array is used instead."""
    tp, rows, pages = _table(table, positions.shape[0], pages)
    _check(load_library().pkv_decode_static(
        pool, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(q_norm_w, torch.bfloat16, "q_norm_w"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(positions, torch.int32, "positions"), tp, rows, pages,
        _dev(out, torch.bfloat16, "out"), _stream(stream)), "pkv_decode_static")


def pkv_step(pool, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, step_positions, table, out, workspace,
             stream=None, pages=None) -> None:
    """step_paged; ``table=None`` with ``pages`` is step_packed over contiguous rows."""
    P = int(positions.shape[0])
    tp, rows, pages = _table(table, step_positions.shape[0], pages)
    _check(load_library().pkv_step(
        pool, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(q_norm_w, torch.bfloat16, "q_norm_w"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(positions, torch.int32, "positions"), _dev(prow, torch.int32, "prow"),
        _dev(slots, torch.int32, "slots", allow_none=True), _dev(step_positions, torch.int32, "step_positions"),
        tp, P, rows, pages, _dev(out, torch.bfloat16, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)), "pkv_step")


def pkv_prefill(pool, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, table, out, workspace, stream=None,
                rows=None, pages=None) -> None:
    """prefill_paged; ``table=None`` with ``rows`` and ``pages`` is prefill over contiguous rows."""
    P = int(positions.shape[0])
    tp, rows, pages = _table(table, rows, pages)
    _check(load_library().pkv_prefill(
        pool, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(q_norm_w, torch.bfloat16, "q_norm_w"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(positions, torch.int32, "positions"), _dev(prow, torch.int32, "prow"),
        _dev(slots, torch.int32, "slots", allow_none=True), tp, P, rows, pages,
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)), "pkv_prefill")


def pkv_linear_workspace_bytes(pool, tokens: int, in_features: int, out_features: int) -> int:
    n = ctypes.c_size_t()
    _check(load_library().pkv_linear_workspace_bytes(pool, int(tokens), int(in_features), int(out_features),
                                                      ctypes.byref(n)), "pkv_linear_workspace_bytes")
    return n.value


def pkv_linear(pool, x, w, y, workspace=None, stream=None) -> None:
    """y = x w^T: x [tokens][in], w [out][in] (nn.Linear layout), y [tokens][out], all bf16."""
    if x.dim() != 2 or w.dim() != 2 or y.dim() != 2 or x.shape[1] != w.shape[1] or y.shape != (x.shape[0], w.shape[0]):
        raise ValueError(f"shapes x {tuple(x.shape)}, w {tuple(w.shape)}, y {tuple(y.shape)} do not match y = x w^T")
    ws = ctypes.c_void_p(None) if workspace is None else _dev(workspace, torch.uint8, "workspace")
    _check(load_library().pkv_linear(
        pool, _dev(x, torch.bfloat16, "x"), _dev(w, torch.bfloat16, "w"), _dev(y, torch.bfloat16, "y"),
        int(x.shape[0]), int(x.shape[1]), int(w.shape[0]), ws, 0 if workspace is None else workspace.numel(),
        _stream(stream)), "pkv_linear")


def pkv_qkv_proj(pool, x, w_qkv, q, k, v, stream=None) -> None:
    """q, k, v = x Wq^T, x Wk^T, x Wv^T with w_qkv = [Wq; Wk; Wv] stacked row-wise (one launch)."""
    tokens, hidden = int(x.shape[0]), int(x.shape[1])
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.shape[0] != tokens:
            raise ValueError(f"{name} has {t.shape[0]} tokens, x has {tokens}")
    if w_qkv.dim() != 2 or w_qkv.shape[1] != hidden or w_qkv.shape[0] != q[0].numel() + k[0].numel() + v[0].numel():
        raise ValueError(f"w_qkv {tuple(w_qkv.shape)} does not stack the q, k, v projections of x {tuple(x.shape)}")
    _check(load_library().pkv_qkv_proj(
        pool, _dev(x, torch.bfloat16, "x"), _dev(w_qkv, torch.bfloat16, "w_qkv"), tokens, hidden,
        _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), _stream(stream)),
        "pkv_qkv_proj")


def pkv_qkv_proj_append(pool, x, w_qkv, q_norm_w, k_norm_w, positions, table, q_hat, stream=None,
                        pages=None) -> None:
    """q/k/v projection of decode rows with QK-norm, RoPE and the k/v append in its epilogue;
    q_hat (fp32 [tokens][heads][head_dim]) receives the normed, roped q."""
    tokens, hidden = int(x.shape[0]), int(x.shape[1])
    tp, rows, pages = _table(table, positions.shape[0], pages)
    if rows != tokens or q_hat.shape[0] != tokens:
        raise ValueError(f"x has {tokens} tokens, positions/table {rows}, q_hat {q_hat.shape[0]}")
    _check(load_library().pkv_qkv_proj_append(
        pool, _dev(x, torch.bfloat16, "x"), _dev(w_qkv, torch.bfloat16, "w_qkv"), tokens, hidden,
        _dev(q_norm_w, torch.bfloat16, "q_norm_w"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(positions, torch.int32, "positions"), tp, pages, _dev(q_hat, torch.float32, "q_hat"),
        _stream(stream)), "pkv_qkv_proj_append")


def pkv_decode_appended(pool, q_hat, positions, table, out, workspace, stream=None, pages=None) -> None:
    """decode_paged's attention after pkv_qkv_proj_append (q prepared, k/v already in the pool)."""
    tp, rows, pages = _table(table, positions.shape[0], pages)
    _check(load_library().pkv_decode_appended(
        pool, _dev(q_hat, torch.float32, "q_hat"), _dev(positions, torch.int32, "positions"), tp, rows, pages,
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)), "pkv_decode_appended")


def pkv_output_gate(pool, out, gate, stream=None) -> None:
    """out *= sigmoid(gate) in place (the gated-attention variant's output gate)."""
    if out.shape != gate.shape:
        raise ValueError(f"gate {tuple(gate.shape)} does not match out {tuple(out.shape)}")
    _check(load_library().pkv_output_gate(pool, _dev(out, torch.bfloat16, "out"), _dev(gate, torch.bfloat16, "gate"),
                                          int(out.shape[0]), _stream(stream)), "pkv_output_gate")


def pkv_check_errors(pool, stream=None) -> int:
    f = ctypes.c_uint32()
    _check(load_library().pkv_check_errors(pool, _stream(stream), ctypes.byref(f)), "pkv_check_errors")
    return f.value


def pkv_set_ctas(pool, ctas: int) -> None:
    _check(load_library().pkv_set_ctas(pool, int(ctas)), "pkv_set_ctas")


def pkv_set_wait_limit(pool, ns: int) -> None:
    _check(load_library().pkv_set_wait_limit(pool, int(ns)), "pkv_set_wait_limit")


def pkv_timer_enable(pool, enable) -> None:
    """enable: False/0 off, True/1 every timed launch, 2 the attention launches only."""
    _check(load_library().pkv_timer_enable(pool, int(enable)), "pkv_timer_enable")


def pkv_timer_read(pool):
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(load_library().pkv_timer_read(pool, ctypes.byref(ms), ctypes.byref(n)), "pkv_timer_read")
    return ms.value, n.value


# ------------------------------------------------------------------ convenience (marshalling only)

class PagedKVPool:
    """A pool over caller-owned K/V torch tensors [kv_heads][num_pages*page_size][head_dim] (bf16)."""

    def __init__(self, K: torch.Tensor, V: torch.Tensor, cfg=None, stream=None):
        c = _cfg(cfg)
        if K.shape != V.shape or K.dim() != 3 or K.shape[0] != c.kv_heads or K.shape[2] != c.head_dim \
                or K.shape[1] % c.page_size:
            raise ValueError(f"K/V must be [kv_heads][num_pages*page_size][head_dim], got {tuple(K.shape)}")
        self.K, self.V, self.cfg = K, V, c
        self.num_pages = K.shape[1] // c.page_size
        self.handle = pkv_pool_wrap(c, self.num_pages, K, V, stream)
        self._ws = None
        self._lws = None

    def workspace(self, rows: int, pages: int, prefill_tokens: int = 0) -> torch.Tensor:
        n = pkv_workspace_bytes(self.handle, rows, pages, prefill_tokens)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.K.device)
        return self._ws

    def decode(self, q, k, v, q_norm_w, k_norm_w, positions, table, out=None, stream=None,
               pages=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        pages = table.shape[1] if table is not None else pages
        ws = self.workspace(positions.shape[0], pages, 0)
        pkv_decode(self.handle, q, k, v, q_norm_w, k_norm_w, positions, table, out, ws, stream, pages=pages)
        return out

    def step(self, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, step_positions, table, out=None,
             stream=None, pages=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        pages = table.shape[1] if table is not None else pages
        ws = self.workspace(step_positions.shape[0], pages, positions.shape[0])
        pkv_step(self.handle, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, step_positions, table, out, ws,
                 stream, pages=pages)
        return out

    def prefill(self, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, table, out=None, stream=None,
                rows=None, pages=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        pages = table.shape[1] if table is not None else pages
        ws = self.workspace(0, pages, positions.shape[0])
        pkv_prefill(self.handle, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, table, out, ws, stream,
                    rows=rows, pages=pages)
        return out

    def linear(self, x, w, y=None, stream=None) -> torch.Tensor:
        """y = x w^T on this pool's device (a projection before or after the attention)."""
        if y is None:
            y = torch.empty(x.shape[0], w.shape[0], dtype=torch.bfloat16, device=x.device)
        n = pkv_linear_workspace_bytes(self.handle, x.shape[0], x.shape[1], w.shape[0])
        ws = None
        if n:
            if self._lws is None or self._lws.numel() < n:
                self._lws = torch.empty(n, dtype=torch.uint8, device=x.device)
            ws = self._lws
        pkv_linear(self.handle, x, w, y, ws, stream)
        return y

    def qkv_proj(self, x, w_qkv, q=None, k=None, v=None, stream=None):
        """q [tokens][heads][head_dim], k and v [tokens][kv_heads][head_dim] from x and the stacked weights."""
        c, n = self.cfg, x.shape[0]
        if q is None:
            q = torch.empty(n, c.heads, c.head_dim, dtype=torch.bfloat16, device=x.device)
        if k is None:
            k = torch.empty(n, c.kv_heads, c.head_dim, dtype=torch.bfloat16, device=x.device)
        if v is None:
            v = torch.empty(n, c.kv_heads, c.head_dim, dtype=torch.bfloat16, device=x.device)
        pkv_qkv_proj(self.handle, x, w_qkv, q, k, v, stream)
        return q, k, v

    def decode_layer_fused(self, x, w_qkv, q_norm_w, k_norm_w, positions, table, out=None, q_hat=None,
                           stream=None, pages=None) -> torch.Tensor:
        """The q/k/v projection with norm, RoPE and append fused in, then the attention."""
        c, n = self.cfg, x.shape[0]
        if q_hat is None:
            q_hat = torch.empty(n, c.heads, c.head_dim, dtype=torch.float32, device=x.device)
        if out is None:
            out = torch.empty(n, c.heads, c.head_dim, dtype=torch.bfloat16, device=x.device)
        pages = table.shape[1] if table is not None else pages
        pkv_qkv_proj_append(self.handle, x, w_qkv, q_norm_w, k_norm_w, positions, table, q_hat, stream, pages=pages)
        ws = self.workspace(n, pages, 0)
        pkv_decode_appended(self.handle, q_hat, positions, table, out, ws, stream, pages=pages)
        return out

    def check_errors(self, stream=None) -> int:
        return pkv_check_errors(self.handle, stream)

    def close(self):
        if self.handle is not None and self.handle.value:
            pkv_pool_free(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
