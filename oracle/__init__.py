"""fp64 CPU oracle for the paged-KV GQA decode step (QK-norm, RoPE, page-slot
append, grouped-query attention over pages).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The
product library (``paged_kv_gqa_qk_gb300``) never imports it, and it never
imports the product library: the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision, one
function per step, each citing the passage of the pages it follows).  This
module compiles it with gcc on first use and marshals numpy arrays to it.
bf16 tensors are passed as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

# Defaults from the Qwen3-8B Nest page: nest.toml [generics] (Heads 32,
# KvHeads 8, HeadDim 128, MaxSeq 40960), attention.linnet (PageSize 64),
# rope.linnet (THETA 1e6), norm.linnet (eps 1e-6).
DEFAULT_CONFIG = dict(heads=32, kv_heads=8, head_dim=128, page_size=64, max_seq=40960,
                      rope_theta=1.0e6, eps=1.0e-6, rotary_dim=128)

ERR_POSITION, ERR_PAGE, ERR_ROW, ERR_SLOT = 1, 2, 4, 8


class OrcConfig(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_seq", ctypes.c_int),
                ("rope_theta", ctypes.c_double), ("eps", ctypes.c_double), ("rotary_dim", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libpkv_oracle.so`` (gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -ffp-contract=off: no fused multiply-adds, so every product and sum
        # is the plain IEEE double operation written in the source.
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        c_u16p, c_i32p, c_dp = P(ctypes.c_uint16), P(ctypes.c_int32), P(ctypes.c_double)
        cfgp = P(OrcConfig)
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_round_bf16.argtypes = [ctypes.c_double]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_round_bf16_array.argtypes = [c_dp, c_u16p, ctypes.c_int64]
        lib.orc_round_bf16_array.restype = None
        lib.orc_qk_norm.argtypes = [cfgp, c_u16p, c_u16p, c_dp]
        lib.orc_qk_norm.restype = None
        lib.orc_rope.argtypes = [cfgp, c_dp, ctypes.c_int]
        lib.orc_rope.restype = None
        lib.orc_page_slot.argtypes = [cfgp, c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_page_slot.restype = ctypes.c_int64
        lib.orc_attend.argtypes = [cfgp, c_u16p, c_u16p, ctypes.c_int64, c_i32p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, c_dp, c_dp]
        lib.orc_attend.restype = None
        lib.orc_attend_split.argtypes = [cfgp, c_u16p, c_u16p, ctypes.c_int64, c_i32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, c_dp, ctypes.c_int,
                                         c_i32p, c_dp]
        lib.orc_attend_split.restype = None
        lib.orc_step.argtypes = [cfgp, c_u16p, c_u16p, ctypes.c_int, c_u16p, c_u16p, c_u16p, c_u16p, c_u16p,
                                 c_i32p, c_i32p, c_i32p, c_i32p, c_i32p, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, c_i32p, ctypes.c_int, c_dp, P(ctypes.c_uint32), ctypes.c_int]
        lib.orc_step.restype = ctypes.c_int
        _lib = lib
        return lib


def _cfg(cfg: dict | None) -> OrcConfig:
    d = dict(DEFAULT_CONFIG)
    if cfg:
        d.update(cfg)
    if cfg and "head_dim" in cfg and "rotary_dim" not in cfg:
        d["rotary_dim"] = d["head_dim"]   # a custom head size rotates all of it unless told otherwise
    if not 0 <= d["rotary_dim"] <= d["head_dim"] or d["rotary_dim"] % 2:
        raise ValueError(f"rotary_dim {d['rotary_dim']} for head_dim {d['head_dim']}")
    return OrcConfig(d["heads"], d["kv_heads"], d["head_dim"], d["page_size"], d["max_seq"],
                     float(d["rope_theta"]), float(d["eps"]), int(d["rotary_dim"]))


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, f"bf16 arrays are passed as uint16 bit patterns, got {a.dtype}"
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray | None:
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ---------------------------------------------------------------- helpers

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (ties to even, one rounding); returns uint16 bits."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty(x.shape, dtype=np.uint16)
    lib.orc_round_bf16_array(_ptr(x, ctypes.c_double), _ptr(y, ctypes.c_uint16), x.size)
    return y


def qk_norm(x_bits: np.ndarray, w_bits: np.ndarray, cfg: dict | None = None) -> np.ndarray:
    """Per-head RMSNorm of one head vector (bf16 bits) with weight (bf16 bits) -> float64."""
    lib = _load()
    c = _cfg(cfg)
    x, w = _u16(x_bits), _u16(w_bits)
    assert x.shape == (c.head_dim,) and w.shape == (c.head_dim,)
    y = np.empty(c.head_dim, dtype=np.float64)
    lib.orc_qk_norm(ctypes.byref(c), _ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16), _ptr(y, ctypes.c_double))
    return y


def rope(y: np.ndarray, pos: int, cfg: dict | None = None) -> np.ndarray:
    """Rotate-half RoPE of one float64 head vector at position ``pos`` (returns a copy)."""
    lib = _load()
    c = _cfg(cfg)
    out = np.ascontiguousarray(np.array(y, dtype=np.float64, copy=True))
    assert out.shape == (c.head_dim,)
    lib.orc_rope(ctypes.byref(c), _ptr(out, ctypes.c_double), int(pos))
    return out


def page_slot(table: np.ndarray, row: int, pos: int, cfg: dict | None = None) -> int:
    lib = _load()
    c = _cfg(cfg)
    t = _i32(table)
    return int(lib.orc_page_slot(ctypes.byref(c), _ptr(t, ctypes.c_int32), t.shape[1], int(row), int(pos)))


def page_slots(table: np.ndarray, rows: np.ndarray, positions: np.ndarray, cfg: dict | None = None) -> np.ndarray:
    """Slots of (row, position) pairs, one oracle call each."""
    return np.array([page_slot(table, r, p, cfg) for r, p in zip(rows, positions)], dtype=np.int32)


def attend(K: np.ndarray, V: np.ndarray, table: np.ndarray, row: int, pos: int, g: int, qhat: np.ndarray,
           cfg: dict | None = None) -> np.ndarray:
    """Attention of one normed+roped query (float64) over row ``row``'s keys 0..pos of kv head g."""
    lib = _load()
    c = _cfg(cfg)
    K, V, t = _u16(K), _u16(V), _i32(table)
    qh = np.ascontiguousarray(np.asarray(qhat, dtype=np.float64))
    out = np.empty(c.head_dim, dtype=np.float64)
    lib.orc_attend(ctypes.byref(c), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16), K.shape[1],
                   _ptr(t, ctypes.c_int32), t.shape[1], int(row), int(pos), int(g), _ptr(qh, ctypes.c_double),
                   _ptr(out, ctypes.c_double))
    return out


def attend_split(K, V, table, row, pos, g, qhat, split, cfg: dict | None = None) -> np.ndarray:
    """Same as :func:`attend`, computed over position ranges ``split`` and merged by log-sum-exp."""
    lib = _load()
    c = _cfg(cfg)
    K, V, t = _u16(K), _u16(V), _i32(table)
    sp = _i32(split)
    qh = np.ascontiguousarray(np.asarray(qhat, dtype=np.float64))
    out = np.empty(c.head_dim, dtype=np.float64)
    lib.orc_attend_split(ctypes.byref(c), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16), K.shape[1],
                         _ptr(t, ctypes.c_int32), t.shape[1], int(row), int(pos), int(g),
                         _ptr(qh, ctypes.c_double), len(sp) - 1, _ptr(sp, ctypes.c_int32),
                         _ptr(out, ctypes.c_double))
    return out


def step(K: np.ndarray, V: np.ndarray, q, k, v, q_norm_w, k_norm_w, positions, prow, slots, step_positions,
         table, cfg: dict | None = None, sel=None, nthreads: int | None = None):
    """``step_paged``: writes every token's k/v into the pools K, V (in place), then attends.

    K, V: uint16 [kv_heads][num_slots][head_dim].  q [P+R][heads][D], k/v
    [P+R][kv_heads][D] (uint16).  positions/prow/slots: int32 [P] (slots may
    be None: derived from the table).  step_positions: int32 [R] (-1 = no
    step).  table: int32 [R][pages].  sel: token indices whose outputs are
    computed (None: all).  Returns (out float64 [P+R][heads][D], err_bits).
    """
    lib = _load()
    c = _cfg(cfg)
    K, V = _u16(K), _u16(V)
    q, k, v = _u16(q), _u16(k), _u16(v)
    qw, kw = _u16(q_norm_w), _u16(k_norm_w)
    t = _i32(table)
    pos_a, prow_a, slots_a = _i32(positions), _i32(prow), _i32(slots)
    sp = _i32(step_positions)
    P = 0 if pos_a is None else int(pos_a.shape[0])
    R = 0 if sp is None else int(sp.shape[0])
    N = P + R
    assert q.shape == (N, c.heads, c.head_dim), q.shape
    assert k.shape == (N, c.kv_heads, c.head_dim) and v.shape == k.shape
    assert K.shape[0] == c.kv_heads and K.shape[2] == c.head_dim and K.shape == V.shape
    num_slots = K.shape[1]
    assert num_slots % c.page_size == 0
    num_pages = num_slots // c.page_size
    assert t.ndim == 2 and t.shape[0] == R
    sel_a = _i32(sel)
    out = np.zeros((N, c.heads, c.head_dim), dtype=np.float64)
    err = ctypes.c_uint32(0)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.orc_step(ctypes.byref(c), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16), num_pages,
                      _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                      _ptr(qw, ctypes.c_uint16), _ptr(kw, ctypes.c_uint16),
                      _ptr(pos_a, ctypes.c_int32), _ptr(prow_a, ctypes.c_int32), _ptr(slots_a, ctypes.c_int32),
                      _ptr(sp, ctypes.c_int32), _ptr(t, ctypes.c_int32), P, R, t.shape[1],
                      _ptr(sel_a, ctypes.c_int32), 0 if sel_a is None else len(sel_a),
                      _ptr(out, ctypes.c_double), ctypes.byref(err), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: malformed step call")
    return out, int(err.value)


def decode(K, V, q, k, v, q_norm_w, k_norm_w, positions, table, cfg: dict | None = None, sel=None,
           nthreads: int | None = None):
    """``decode_paged``: step with no prompt tokens. Returns (out [R][heads][D] float64, err_bits)."""
    return step(K, V, q, k, v, q_norm_w, k_norm_w, None, None, None, positions, table, cfg=cfg, sel=sel,
                nthreads=nthreads)


def linear(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """A projection without bias, y[t][o] = sum_k x[t][k] w[o][k] (qwen3-8b Nest files,
    src/attention.linnet: q_proj / k_proj / v_proj / o_proj), in float64 on the exact
    values of bf16 x [tokens][in] and w [out][in]; a library matrix product is the step."""
    return bf16_to_f64(_u16(x_bits)) @ bf16_to_f64(_u16(w_bits)).T


def output_gate(out: np.ndarray, gate_bits: np.ndarray) -> np.ndarray:
    """The output gate of the gated attention variant (fantasma model.zig,
    fullAttentionForward: attn_out *= sigmoid(gate)), elementwise in float64 on
    the attention output and the exact values of the bf16 gate."""
    g = bf16_to_f64(_u16(gate_bits))
    return np.asarray(out, dtype=np.float64) / (1.0 + np.exp(-g))
