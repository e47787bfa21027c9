"""fp64 CPU oracle for exact scaled-dot-product attention (fwd + bwd).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The product library never imports it and shares no code with
it; the two meet only in the seeded input generators of ``fa_inputs``.

The arithmetic lives in ``fa_oracle.c`` (plain C, IEEE double, libm exp/log).
This module compiles it with gcc on first use and marshals numpy arrays.

What each function follows:

* ``forward``: the attention definition in "What is Flash Attention?"
  (transcript 01:04: S = QK^T/sqrt(d), row softmax, O = PV) with the safe
  softmax of "Atencao exata, acelerada por nunca escrever a grade gigante."
  (softmax formula with m = max_j x_j); the stored statistic is
  lse = m + ln l, the pair (m, l) kept per row (transcript 06:52).
* ``backward``: the plain chain rule through that definition (the pages state
  only that gradients are exact and that P is recomputed, transcript
  06:52-07:24 and 08:26).
* ``online_softmax`` / ``online_attention_row``: the running-max update of
  transcript 04:46-05:17, used only to pin online == two-pass.
* ``decode``: the same definition for Nq query rows against an Nk-row key /
  value cache (the transcript's closing mention of KV caches, 11:33), query i
  at cache position Nk - Nq + i for the causal mask.
* ``mask=`` (block-sparse, the talk's block-sparse FlashAttention): scores of
  dropped (query block, key block) pairs are -inf; a row with no visible key
  is defined as o = 0, lse = -inf with zero gradients.
* ``dropout=(p, seed, offset)`` (the talk's dropout on P before the product
  with V, transcript Q&A after 10:00): O = (P o Z / (1 - p)) V, lse that of
  P.  Z is drawn by Philox4x32-10 (Salmon et al., SC 2011) at counter
  (j // 8, i, bh, offset) with key seed: key j takes the low (even j) or
  high (odd j) 16 bits of word (j // 2) % 4, and is kept iff they are
  >= floor(p * 2^16); kept values are scaled by the inverse keep probability.

Parity of every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libfa_oracle.so")
_lock = threading.Lock()
_default = None


def compile_library(src: str, out: str) -> str:
    """Compile a copy of the oracle's C source into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so every product and sum is a
    # separately rounded IEEE double operation, identical on x86 and Arm.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into oracle/_build/libfa_oracle.so (gcc, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_library(SOURCE, _LIB_PATH)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (bf16 -> f64 is exact)."""
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _sel(rows, BH: int, N: int):
    if rows is None:
        return None, BH * N
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    if r.size and (r.min() < 0 or r.max() >= BH * N):
        raise ValueError("row index out of range")
    return r, int(r.size)


def _shape(q):
    if q.ndim == 4:
        B, H, N, d = q.shape
        return B * H, N, d
    if q.ndim == 3:
        BH, N, d = q.shape
        return BH, N, d
    raise ValueError("expected [B,H,N,d] or [BH,N,d]")


class Oracle:
    """The oracle bound to one compiled copy of fa_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        lib.fa_oracle_forward.argtypes = [dp, dp, dp, i, i, i, d, i, ip, i64, dp, dp, i]
        lib.fa_oracle_backward_rows.argtypes = [dp, dp, dp, dp, i, i, i, d, i, ip, i64,
                                                dp, dp, dp, dp, dp, i]
        lib.fa_oracle_backward_cols.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, d, i,
                                                ip, i64, dp, dp, i]
        lib.fa_oracle_online_softmax.argtypes = [dp, i, i, dp, dp]
        lib.fa_oracle_online_attention_row.argtypes = [dp, dp, i, i, i, dp, dp]
        lib.fa_oracle_decode.argtypes = [dp, dp, dp, i, i, i, i, d, i, dp, dp, i]
        lib.fa_oracle_decode.restype = ctypes.c_int
        lib.fa_oracle_set_block_mask.argtypes = [ctypes.c_void_p, i, i, i, i64]
        lib.fa_oracle_set_block_mask.restype = None
        lib.fa_oracle_set_dropout.argtypes = [i, ctypes.c_uint64, ctypes.c_uint32,
                                              ctypes.c_uint32, d]
        lib.fa_oracle_set_dropout.restype = None
        lib.fa_oracle_dropout_u16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, i64, i, i]
        lib.fa_oracle_dropout_u16.restype = ctypes.c_uint32
        lib.fa_oracle_philox4x32_10.argtypes = [ctypes.c_void_p] * 3
        lib.fa_oracle_philox4x32_10.restype = None
        for f in (lib.fa_oracle_forward, lib.fa_oracle_backward_rows,
                  lib.fa_oracle_backward_cols, lib.fa_oracle_online_softmax,
                  lib.fa_oracle_online_attention_row):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def _masked(self, mask, block, BH, dropout=None):
        """Context manager that installs a block mask and / or dropout for the
        calls inside it.

        mask: uint8 array [nqb, nkb] (shared by every (b,h)) or [BH, nqb, nkb];
        nonzero keeps the (query block, key block) pair.  block = (bq, bk) rows.
        dropout: None or (p, seed, offset); see ``dropout_params``.
        """
        lib = self.lib

        class _Ctx:
            def __enter__(ctx):
                if dropout is not None:
                    pd, seed, offset = dropout
                    thr, rs = dropout_params(pd)
                    lib.fa_oracle_set_dropout(1, int(seed) & (2**64 - 1),
                                              int(offset) & 0xFFFFFFFF, thr, rs)
                if mask is None:
                    return ctx
                m = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
                if m.ndim == 2:
                    m = m[None]
                if m.shape[0] not in (1, BH):
                    raise ValueError("mask must be [nqb, nkb] or [BH, nqb, nkb]")
                ctx.m = m
                stride = 0 if m.shape[0] == 1 else m.shape[1] * m.shape[2]
                lib.fa_oracle_set_block_mask(m.ctypes.data, int(block[0]), int(block[1]),
                                             int(m.shape[2]), int(stride))
                return ctx

            def __exit__(ctx, *exc):
                lib.fa_oracle_set_block_mask(None, 1, 1, 0, 0)
                lib.fa_oracle_set_dropout(0, 0, 0, 0, 1.0)
                return False

        return _Ctx()

    def forward(self, q, k, v, scale: float, causal: bool, rows=None,
                nthreads: int | None = None, mask=None, block=(128, 128), dropout=None):
        """O and lse of the definition.

        q, k, v: [B,H,N,d] or [BH,N,d] (any dtype; converted exactly to float64).
        rows: None for every row, else flat indices bh*N + i.
        Returns (o, lse): o is [BH*N, d] (or [len(rows), d]), lse [BH*N] (or [len(rows)]).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        BH, N, d = _shape(q)
        sel, n = _sel(rows, BH, N)
        o = np.empty((n, d), np.float64)
        lse = np.empty((n,), np.float64)
        with self._masked(mask, block, BH, dropout):
            rc = self.lib.fa_oracle_forward(
                _ptr(q), _ptr(k), _ptr(v), BH, N, d, float(scale), int(bool(causal)),
                _iptr(sel), n, _ptr(o), _ptr(lse), int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"fa_oracle_forward failed ({rc})")
        return o, lse

    def backward_rows(self, q, k, v, dO, scale: float, causal: bool, rows=None,
                      nthreads: int | None = None, mask=None, block=(128, 128),
                      dropout=None):
        """Row pass: dq for the selected rows plus per-row m, l, D and D_alt.

        D is sum_j P_ij dP_ij; D_alt is sum_c dO_ic O_ic.  They agree exactly in
        real arithmetic; the pins check they agree to fp64 rounding.
        """
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        BH, N, d = _shape(q)
        sel, n = _sel(rows, BH, N)
        dq = np.empty((n, d), np.float64)
        m = np.empty((n,), np.float64)
        l = np.empty((n,), np.float64)
        D = np.empty((n,), np.float64)
        D_alt = np.empty((n,), np.float64)
        with self._masked(mask, block, BH, dropout):
            rc = self.lib.fa_oracle_backward_rows(
                _ptr(q), _ptr(k), _ptr(v), _ptr(dO), BH, N, d, float(scale), int(bool(causal)),
                _iptr(sel), n, _ptr(dq), _ptr(m), _ptr(l), _ptr(D), _ptr(D_alt),
                int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"fa_oracle_backward_rows failed ({rc})")
        return dq, m, l, D, D_alt

    def backward_cols(self, q, k, v, dO, m_all, l_all, D_all, scale: float, causal: bool,
                      cols=None, nthreads: int | None = None, mask=None, block=(128, 128),
                      dropout=None):
        """Column pass: dk, dv for the selected key rows (flat bh*N + j).

        m_all, l_all, D_all must cover every row (from backward_rows(rows=None)).
        """
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        m_all, l_all, D_all = _f64(m_all), _f64(l_all), _f64(D_all)
        BH, N, d = _shape(q)
        if m_all.size != BH * N or l_all.size != BH * N or D_all.size != BH * N:
            raise ValueError("m_all, l_all, D_all must hold every row")
        sel, n = _sel(cols, BH, N)
        dk = np.empty((n, d), np.float64)
        dv = np.empty((n, d), np.float64)
        with self._masked(mask, block, BH, dropout):
            rc = self.lib.fa_oracle_backward_cols(
                _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(m_all), _ptr(l_all), _ptr(D_all),
                BH, N, d, float(scale), int(bool(causal)), _iptr(sel), n, _ptr(dk), _ptr(dv),
                int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"fa_oracle_backward_cols failed ({rc})")
        return dk, dv

    def backward(self, q, k, v, dO, scale: float, causal: bool, nthreads: int | None = None,
                 mask=None, block=(128, 128), dropout=None):
        """Full backward: (dq, dk, dv) each [BH*N, d], plus (m, l, D, D_alt) per row."""
        dq, m, l, D, D_alt = self.backward_rows(q, k, v, dO, scale, causal, None, nthreads,
                                                mask=mask, block=block, dropout=dropout)
        dk, dv = self.backward_cols(q, k, v, dO, m, l, D, scale, causal, None, nthreads,
                                    mask=mask, block=block, dropout=dropout)
        return dq, dk, dv, (m, l, D, D_alt)

    def decode(self, q, k, v, scale: float, causal: bool, nthreads: int | None = None):
        """A few queries against a key/value cache: q [..., Nq, d], k, v [..., Nk, d].

        Query i sits at cache position Nk - Nq + i; with causal it sees keys up
        to that position.  Returns (o [BH*Nq, d], lse [BH*Nq]).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        d = q.shape[-1]
        Nq, Nk = q.shape[-2], k.shape[-2]
        BH = int(np.prod(q.shape[:-2]))
        if k.shape != v.shape or int(np.prod(k.shape[:-2])) != BH or k.shape[-1] != d:
            raise ValueError("q, k, v shapes disagree")
        o = np.empty((BH * Nq, d), np.float64)
        lse = np.empty((BH * Nq,), np.float64)
        rc = self.lib.fa_oracle_decode(_ptr(q), _ptr(k), _ptr(v), BH, Nq, Nk, d, float(scale),
                                       int(bool(causal)), _ptr(o), _ptr(lse),
                                       int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"fa_oracle_decode failed ({rc})")
        return o, lse

    def philox(self, ctr, key):
        """Philox4x32-10 of a 4-word counter and a 2-word key (4 words out)."""
        c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
        kk = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
        if c.shape != (4,) or kk.shape != (2,):
            raise ValueError("counter has 4 words, key 2")
        out = np.zeros(4, np.uint32)
        self.lib.fa_oracle_philox4x32_10(c.ctypes.data, kk.ctypes.data, out.ctypes.data)
        return [int(x) for x in out]

    def dropout_u16(self, seed: int, offset: int, bh: int, i: int, j: int) -> int:
        """The 16-bit uniform that decides element (i, j) of head bh."""
        return int(self.lib.fa_oracle_dropout_u16(int(seed) & (2**64 - 1),
                                                  int(offset) & 0xFFFFFFFF, int(bh),
                                                  int(i), int(j)))

    def dropout_keep(self, p: float, seed: int, offset: int, bh: int, n_rows: int, n_cols: int):
        """Keep matrix Z [n_rows, n_cols] (bool) of head bh."""
        thr, _ = dropout_params(p)
        z = np.empty((n_rows, n_cols), dtype=bool)
        for i in range(n_rows):
            for j in range(n_cols):
                z[i, j] = self.dropout_u16(seed, offset, bh, i, j) >= thr
        return z

    def online_softmax(self, x, block: int):
        """Running (m, l) after each block of the row x (online update)."""
        x = _f64(x).reshape(-1)
        nb = -(-x.size // block)
        m = np.empty((nb,), np.float64)
        l = np.empty((nb,), np.float64)
        rc = self.lib.fa_oracle_online_softmax(_ptr(x), x.size, int(block), _ptr(m), _ptr(l))
        if rc != nb:
            raise RuntimeError(f"fa_oracle_online_softmax failed ({rc})")
        return m, l

    def online_attention_row(self, s, v, block: int):
        """One attention row by the online update: (o [d], lse)."""
        s = _f64(s).reshape(-1)
        v = _f64(v)
        n, d = v.shape
        if s.size != n:
            raise ValueError("s and v disagree on n")
        o = np.empty((d,), np.float64)
        lse = np.empty((1,), np.float64)
        rc = self.lib.fa_oracle_online_attention_row(_ptr(s), _ptr(v), n, d, int(block),
                                                     _ptr(o), _ptr(lse))
        if rc != 0:
            raise RuntimeError(f"fa_oracle_online_attention_row failed ({rc})")
        return o, float(lse[0])


def dropout_params(p: float):
    """(thr, rs) of a dropout probability p in [0, 1).

    p is first rounded to IEEE single (the precision the library takes it
    in); an element is kept iff its 16-bit uniform is >= thr = floor(p * 2^16),
    so it is kept with probability (65536 - thr) / 65536, and kept values are
    scaled by the inverse of that, rs = 65536 / (65536 - thr).
    """
    p32 = float(np.float32(p))
    if not 0.0 <= p32 < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    thr = int(np.floor(p32 * 65536.0))
    return thr, 65536.0 / (65536.0 - thr)


def default() -> Oracle:
    """The oracle compiled from oracle/fa_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def forward(*a, **kw):
    return default().forward(*a, **kw)


def backward_rows(*a, **kw):
    return default().backward_rows(*a, **kw)


def backward_cols(*a, **kw):
    return default().backward_cols(*a, **kw)


def backward(*a, **kw):
    return default().backward(*a, **kw)


def online_softmax(*a, **kw):
    return default().online_softmax(*a, **kw)


def decode(*a, **kw):
    return default().decode(*a, **kw)


def online_attention_row(*a, **kw):
    return default().online_attention_row(*a, **kw)


def dropout_u16(*a, **kw):
    return default().dropout_u16(*a, **kw)


def dropout_keep(*a, **kw):
    return default().dropout_keep(*a, **kw)
