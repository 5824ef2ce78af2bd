"""FP64 CPU oracle for the attention leaf — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
import this package.  The product path (``non_causal_prefix_gb300``) never
does, and this package never imports the product path.

The arithmetic lives in ``attn_oracle.c`` (dense and prefix-cached forms),
``attn_oracle_block_causal.c`` and ``attn_oracle_masked_prefix.c`` (plain C,
FP64, OpenMP over output rows); this module only compiles them with gcc into
one library and marshals numpy arrays.
Inputs are bf16 bit patterns (``numpy.uint16``, layout ``[B, N, H, D]``);
outputs are float64 ``[B, Nq, H, D]`` (or ``[rows, D]`` for sampled rows).

Pins: the dense and prefix functions are checked in ``tests/test_oracle.py``,
the block-causal ones in ``tests/test_oracle_block_causal.py``, the masked
prefix ones in ``tests/test_oracle_masked_prefix.py``, against
closed forms (one key; identical keys; one dominant logit; the two-key
logistic weight), invariants (joint K/V permutation, query/head/batch
independence, prefix == dense on the explicit concatenation), a pure-Python
brute force on tiny shapes and float64 ``torch.softmax`` on small ones.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
SOURCE_BLOCK_CAUSAL = os.path.join(_HERE, "attn_oracle_block_causal.c")
SOURCE_MASKED_PREFIX = os.path.join(_HERE, "attn_oracle_masked_prefix.c")
SOURCES = [SOURCE, SOURCE_BLOCK_CAUSAL, SOURCE_MASKED_PREFIX]
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off"]


def compile_source(src, out: str) -> str:
    """Compile C source(s) of the oracle (a path or a list) into a shared library at ``out``."""
    srcs = [src] if isinstance(src, str) else list(src)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, *srcs, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) if stale."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in SOURCES)):
        return _LIB
    return compile_source(SOURCES, _LIB)


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16)")
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with status {rc}")


class Oracle:
    """The oracle's entry points, bound to one compiled library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ci = ctypes.c_int
        lib.oracle_dense_attention.argtypes = [u16p, u16p, u16p, f64p, ci, ci, ci, ci, ci]
        lib.oracle_dense_attention_rows.argtypes = [
            u16p, u16p, u16p, f64p, ci, ci, ci, ci, ci, i64p, ctypes.c_int64]
        lib.oracle_prefix_attention.argtypes = [
            u16p, u16p, u16p, u16p, u16p, f64p, ci, ci, ci, ci, ci, ci]
        lib.oracle_prefix_attention_rows.argtypes = [
            u16p, u16p, u16p, u16p, u16p, f64p, ci, ci, ci, ci, ci, ci, i64p, ctypes.c_int64]
        for f in ("oracle_dense_attention", "oracle_dense_attention_rows",
                  "oracle_prefix_attention", "oracle_prefix_attention_rows",
                  "oracle_max_threads"):
            getattr(lib, f).restype = ci
        # The block-causal form lives in its own source; a library built from
        # attn_oracle.c alone (the tests' single-file mutants) lacks it.
        if hasattr(lib, "oracle_block_causal_attention"):
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_block_causal_attention.argtypes = [
                u16p, u16p, u16p, i32p, f64p, ci, ci, ci, ci]
            lib.oracle_block_causal_attention_rows.argtypes = [
                u16p, u16p, u16p, i32p, f64p, ci, ci, ci, ci, i64p, ctypes.c_int64]
            lib.oracle_block_causal_attention.restype = ci
            lib.oracle_block_causal_attention_rows.restype = ci
        if hasattr(lib, "oracle_masked_prefix_attention"):
            i32p = ctypes.POINTER(ctypes.c_int32)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            cf = ctypes.c_float
            lib.oracle_masked_prefix_attention.argtypes = [
                u16p, u16p, u16p, u16p, u16p, i32p, u8p, cf, f64p, ci, ci, ci, ci, ci]
            lib.oracle_masked_prefix_attention_rows.argtypes = [
                u16p, u16p, u16p, u16p, u16p, i32p, u8p, cf, f64p, ci, ci, ci, ci, ci, i64p,
                ctypes.c_int64]
            lib.oracle_masked_prefix_attention.restype = ci
            lib.oracle_masked_prefix_attention_rows.restype = ci
        lib.oracle_set_threads.argtypes = [ci]
        lib.oracle_set_threads.restype = None
        self.lib = lib
        self.path = lib_path

    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def dense_attention(self, Q, K, V) -> np.ndarray:
        """softmax(Q K^T * D^-0.5) V in FP64; Q [B,Nq,H,D], K/V [B,Nk,H,D]."""
        Q, K, V = _u16(Q), _u16(K), _u16(V)
        B, Nq, H, D = Q.shape
        Nk = K.shape[1]
        if K.shape != (B, Nk, H, D) or V.shape != K.shape:
            raise ValueError("K and V must be [B, Nk, H, D] with Q's B, H, D")
        out = np.empty((B, Nq, H, D), dtype=np.float64)
        _check(self.lib.oracle_dense_attention(
            _ptr(Q, ctypes.c_uint16), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16),
            _ptr(out, ctypes.c_double), B, Nq, Nk, H, D), "oracle_dense_attention")
        return out

    def dense_attention_rows(self, Q, K, V, rows) -> np.ndarray:
        """Sampled rows of ``dense_attention``: flat row r = (b*Nq + i)*H + h."""
        Q, K, V = _u16(Q), _u16(K), _u16(V)
        B, Nq, H, D = Q.shape
        Nk = K.shape[1]
        if K.shape != (B, Nk, H, D) or V.shape != K.shape:
            raise ValueError("K and V must be [B, Nk, H, D] with Q's B, H, D")
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.size, D), dtype=np.float64)
        _check(self.lib.oracle_dense_attention_rows(
            _ptr(Q, ctypes.c_uint16), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16),
            _ptr(out, ctypes.c_double), B, Nq, Nk, H, D, _ptr(rows, ctypes.c_int64),
            rows.size), "oracle_dense_attention_rows")
        return out

    @staticmethod
    def _prefix_args(Q, Kp, Vp, Kc, Vc):
        Q, Kc, Vc = _u16(Q), _u16(Kc), _u16(Vc)
        B, Nq, H, D = Q.shape
        Nc = Kc.shape[1]
        Np = 0 if Kp is None else Kp.shape[1]
        if Np > 0:
            Kp, Vp = _u16(Kp), _u16(Vp)
            if Kp.shape != (B, Np, H, D) or Vp.shape != Kp.shape:
                raise ValueError("K_prefix/V_prefix must be [B, Np, H, D]")
            pk, pv = _ptr(Kp, ctypes.c_uint16), _ptr(Vp, ctypes.c_uint16)
        else:
            pk = pv = ctypes.POINTER(ctypes.c_uint16)()
        if Kc.shape != (B, Nc, H, D) or Vc.shape != Kc.shape:
            raise ValueError("K_current/V_current must be [B, Nc, H, D]")
        return (Q, Kp, Vp, Kc, Vc), (pk, pv), (B, Nq, Np, Nc, H, D)

    def prefix_attention(self, Q, K_prefix, V_prefix, K_current, V_current) -> np.ndarray:
        """Q attends to cat(K_prefix, K_current) / cat(V_prefix, V_current), FP64."""
        keep, (pk, pv), (B, Nq, Np, Nc, H, D) = self._prefix_args(
            Q, K_prefix, V_prefix, K_current, V_current)
        Q, _, _, Kc, Vc = keep
        out = np.empty((B, Nq, H, D), dtype=np.float64)
        _check(self.lib.oracle_prefix_attention(
            _ptr(Q, ctypes.c_uint16), pk, pv, _ptr(Kc, ctypes.c_uint16),
            _ptr(Vc, ctypes.c_uint16), _ptr(out, ctypes.c_double), B, Nq, Np, Nc, H, D),
            "oracle_prefix_attention")
        return out

    def prefix_attention_rows(self, Q, K_prefix, V_prefix, K_current, V_current,
                              rows) -> np.ndarray:
        """Sampled rows of ``prefix_attention`` (flat row r = (b*Nq + i)*H + h)."""
        keep, (pk, pv), (B, Nq, Np, Nc, H, D) = self._prefix_args(
            Q, K_prefix, V_prefix, K_current, V_current)
        Q, _, _, Kc, Vc = keep
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.size, D), dtype=np.float64)
        _check(self.lib.oracle_prefix_attention_rows(
            _ptr(Q, ctypes.c_uint16), pk, pv, _ptr(Kc, ctypes.c_uint16),
            _ptr(Vc, ctypes.c_uint16), _ptr(out, ctypes.c_double), B, Nq, Np, Nc, H, D,
            _ptr(rows, ctypes.c_int64), rows.size), "oracle_prefix_attention_rows")
        return out

    def block_causal_attention(self, Q, K, V, image_ids) -> np.ndarray:
        """Block-causal self-attention in FP64: query i sees key j iff j <= i or
        both carry the same image id >= 0.  Q/K/V [B,N,H,D], image_ids [N]."""
        Q, K, V = _u16(Q), _u16(K), _u16(V)
        B, N, H, D = Q.shape
        if K.shape != Q.shape or V.shape != Q.shape:
            raise ValueError("Q, K, V must all be [B, N, H, D]")
        ids = np.ascontiguousarray(image_ids, dtype=np.int32)
        if ids.shape != (N,):
            raise ValueError("image_ids must be [N]")
        out = np.empty((B, N, H, D), dtype=np.float64)
        _check(self.lib.oracle_block_causal_attention(
            _ptr(Q, ctypes.c_uint16), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16),
            _ptr(ids, ctypes.c_int32), _ptr(out, ctypes.c_double), B, N, H, D),
            "oracle_block_causal_attention")
        return out

    def block_causal_attention_rows(self, Q, K, V, image_ids, rows) -> np.ndarray:
        """Sampled rows of ``block_causal_attention`` (flat row r = (b*N + i)*H + h)."""
        Q, K, V = _u16(Q), _u16(K), _u16(V)
        B, N, H, D = Q.shape
        if K.shape != Q.shape or V.shape != Q.shape:
            raise ValueError("Q, K, V must all be [B, N, H, D]")
        ids = np.ascontiguousarray(image_ids, dtype=np.int32)
        if ids.shape != (N,):
            raise ValueError("image_ids must be [N]")
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.size, D), dtype=np.float64)
        _check(self.lib.oracle_block_causal_attention_rows(
            _ptr(Q, ctypes.c_uint16), _ptr(K, ctypes.c_uint16), _ptr(V, ctypes.c_uint16),
            _ptr(ids, ctypes.c_int32), _ptr(out, ctypes.c_double), B, N, H, D,
            _ptr(rows, ctypes.c_int64), rows.size), "oracle_block_causal_attention_rows")
        return out

    def _masked_prefix_args(self, Q, K_current, V_current, K_prefix, V_prefix, image_ids,
                            key_valid):
        Q, Kc, Vc = _u16(Q), _u16(K_current), _u16(V_current)
        B, Nq, H, D = Q.shape
        if Kc.shape != Q.shape or Vc.shape != Q.shape:
            raise ValueError("Q, K_current, V_current must all be [B, Nq, H, D]")
        Np = 0 if K_prefix is None else K_prefix.shape[1]
        if Np > 0:
            Kp, Vp = _u16(K_prefix), _u16(V_prefix)
            if Kp.shape != (B, Np, H, D) or Vp.shape != Kp.shape:
                raise ValueError("K_prefix/V_prefix must be [B, Np, H, D]")
            pk, pv = _ptr(Kp, ctypes.c_uint16), _ptr(Vp, ctypes.c_uint16)
        else:
            Kp = Vp = None
            pk = pv = ctypes.POINTER(ctypes.c_uint16)()
        ids = np.ascontiguousarray(image_ids, dtype=np.int32)
        valid = np.ascontiguousarray(key_valid, dtype=np.uint8)
        if ids.shape != (Np + Nq,) or valid.shape != (B, Np + Nq):
            raise ValueError("image_ids must be [Np + Nq] and key_valid [B, Np + Nq]")
        keep = (Q, Kc, Vc, Kp, Vp, ids, valid)
        return keep, (pk, pv), (B, Nq, Np, H, D)

    def masked_prefix_attention(self, Q, K_current, V_current, K_prefix, V_prefix, image_ids,
                                key_valid, sm_scale) -> np.ndarray:
        """Masked prefix-cached attention in FP64 (the pre-audit prefix form)."""
        keep, (pk, pv), (B, Nq, Np, H, D) = self._masked_prefix_args(
            Q, K_current, V_current, K_prefix, V_prefix, image_ids, key_valid)
        Q, Kc, Vc, _, _, ids, valid = keep
        out = np.empty((B, Nq, H, D), dtype=np.float64)
        _check(self.lib.oracle_masked_prefix_attention(
            _ptr(Q, ctypes.c_uint16), _ptr(Kc, ctypes.c_uint16), _ptr(Vc, ctypes.c_uint16), pk, pv,
            _ptr(ids, ctypes.c_int32), _ptr(valid, ctypes.c_uint8), float(sm_scale),
            _ptr(out, ctypes.c_double), B, Nq, Np, H, D), "oracle_masked_prefix_attention")
        return out

    def masked_prefix_attention_rows(self, Q, K_current, V_current, K_prefix, V_prefix, image_ids,
                                     key_valid, sm_scale, rows) -> np.ndarray:
        """Sampled rows of ``masked_prefix_attention`` (flat row r = (b*Nq + i)*H + h)."""
        keep, (pk, pv), (B, Nq, Np, H, D) = self._masked_prefix_args(
            Q, K_current, V_current, K_prefix, V_prefix, image_ids, key_valid)
        Q, Kc, Vc, _, _, ids, valid = keep
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.size, D), dtype=np.float64)
        _check(self.lib.oracle_masked_prefix_attention_rows(
            _ptr(Q, ctypes.c_uint16), _ptr(Kc, ctypes.c_uint16), _ptr(Vc, ctypes.c_uint16), pk, pv,
            _ptr(ids, ctypes.c_int32), _ptr(valid, ctypes.c_uint8), float(sm_scale),
            _ptr(out, ctypes.c_double), B, Nq, Np, H, D, _ptr(rows, ctypes.c_int64), rows.size),
            "oracle_masked_prefix_attention_rows")
        return out


def default() -> Oracle:
    """The oracle compiled from ``attn_oracle.c`` (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def set_threads(n: int) -> None:
    default().set_threads(n)


def max_threads() -> int:
    return default().max_threads()


def dense_attention(Q, K, V) -> np.ndarray:
    return default().dense_attention(Q, K, V)


def dense_attention_rows(Q, K, V, rows) -> np.ndarray:
    return default().dense_attention_rows(Q, K, V, rows)


def prefix_attention(Q, K_prefix, V_prefix, K_current, V_current) -> np.ndarray:
    return default().prefix_attention(Q, K_prefix, V_prefix, K_current, V_current)


def prefix_attention_rows(Q, K_prefix, V_prefix, K_current, V_current, rows) -> np.ndarray:
    return default().prefix_attention_rows(Q, K_prefix, V_prefix, K_current, V_current, rows)


def block_causal_attention(Q, K, V, image_ids) -> np.ndarray:
    return default().block_causal_attention(Q, K, V, image_ids)


def block_causal_attention_rows(Q, K, V, image_ids, rows) -> np.ndarray:
    return default().block_causal_attention_rows(Q, K, V, image_ids, rows)


def masked_prefix_attention(Q, K_current, V_current, K_prefix, V_prefix, image_ids, key_valid,
                            sm_scale) -> np.ndarray:
    return default().masked_prefix_attention(Q, K_current, V_current, K_prefix, V_prefix,
                                             image_ids, key_valid, sm_scale)


def masked_prefix_attention_rows(Q, K_current, V_current, K_prefix, V_prefix, image_ids, key_valid,
                                 sm_scale, rows) -> np.ndarray:
    return default().masked_prefix_attention_rows(Q, K_current, V_current, K_prefix, V_prefix,
                                                  image_ids, key_valid, sm_scale, rows)
