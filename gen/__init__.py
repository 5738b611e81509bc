"""Seeded synthetic inputs for the DSA decode/prefill workloads.

The random source and layout helpers live in ``gen.c`` (SplitMix64, Irwin-Hall normals, Fisher-Yates
permutations, OCP E4M3 encoding for FP8 inputs).  This module only loads that library; the workload
recipes are in :mod:`gen.workloads`.  Nothing here computes indexer scores, Top-K or attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_gen.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into libdsa_gen.so (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            vp = ctypes.c_void_p
            L.dsa_gen_draw.restype = u64
            L.dsa_gen_draw.argtypes = [u64, u64]
            L.dsa_gen_stream_key.restype = u64
            L.dsa_gen_stream_key.argtypes = [u64, u64]
            L.dsa_gen_normal_bf16.argtypes = [u64, u64, i64, f32, vp]
            L.dsa_gen_uniform_f32.argtypes = [u64, u64, i64, f32, f32, vp]
            L.dsa_gen_uniform_int.argtypes = [u64, u64, i64, i64, i64, vp]
            L.dsa_gen_permutation.argtypes = [u64, i32, vp]
            L.dsa_gen_sample_without_replacement.restype = ctypes.c_int
            L.dsa_gen_sample_without_replacement.argtypes = [u64, i32, i32, vp]
            L.dsa_gen_paged_normal_bf16.argtypes = [u64, i32, vp, vp, i32, i32, i32, i64, f32, vp]
            L.dsa_gen_e4m3_encode.restype = ctypes.c_uint8
            L.dsa_gen_e4m3_encode.argtypes = [f32]
            L.dsa_gen_quantize_e4m3_rows.argtypes = [vp, i64, i32, vp, vp]
            L.dsa_gen_e4m3_encode_array.argtypes = [vp, i64, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def stream_key(seed: int, tensor_id: int) -> int:
    return int(lib().dsa_gen_stream_key(seed & (2**64 - 1), tensor_id))


def draw(key: int, i: int) -> int:
    return int(lib().dsa_gen_draw(key, i))


def normal_bf16(key: int, n: int, offset: int = 0, scale: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().dsa_gen_normal_bf16(key, offset, n, scale, _ptr(out))
    return out


def uniform_f32(key: int, n: int, lo: float = 0.0, hi: float = 1.0, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().dsa_gen_uniform_f32(key, offset, n, lo, hi, _ptr(out))
    return out


def uniform_int(key: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    lib().dsa_gen_uniform_int(key, offset, n, lo, hi, _ptr(out))
    return out


def permutation(key: int, n: int) -> np.ndarray:
    out = np.empty(max(n, 1), dtype=np.int32)
    lib().dsa_gen_permutation(key, n, _ptr(out))
    return out[:n]


def sample_without_replacement(key: int, n: int, m: int) -> np.ndarray:
    out = np.empty(max(m, 1), dtype=np.int32)
    rc = lib().dsa_gen_sample_without_replacement(key, n, m, _ptr(out))
    if rc != 0:
        raise ValueError(f"sample_without_replacement({n}, {m}) failed: {rc}")
    return out[:m]


def paged_normal_bf16(key, seq_lens, page_table, page_size, width, row_stride_b, num_pages, scale=1.0):
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    cache = np.zeros((num_pages, page_size, width), dtype=np.uint16)
    lib().dsa_gen_paged_normal_bf16(key, len(seq_lens), _ptr(seq_lens), _ptr(page_table), page_table.shape[1],
                                    page_size, width, row_stride_b, scale, _ptr(cache))
    return cache


def e4m3_encode(v: float) -> int:
    return int(lib().dsa_gen_e4m3_encode(v))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().dsa_gen_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def quantize_e4m3_rows(x_bf16: np.ndarray):
    """Row-wise absmax/448 quantisation of a bf16-bits array [..., cols] -> (codes u8, scales f32[...])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    cols = x.shape[-1]
    rows = x.size // cols
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    lib().dsa_gen_quantize_e4m3_rows(_ptr(x), rows, cols, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_mx_rows(x_bf16: np.ndarray, group: int = 32):
    """MX (OCP microscaling) E4M3 quantisation of a bf16-bits array [..., cols] with one E8M0 scale per
    `group` consecutive elements: shared exponent floor(log2(absmax)) - 8 (the largest E4M3 exponent),
    clamped to the E8M0 range; codes = E4M3(x / 2^shared) with saturation; an all-zero group gets
    exponent 0 (byte 127).  Returns (codes uint8 [..., cols], scale bytes uint8 [..., cols / group])."""
    x = bf16_to_f32(np.ascontiguousarray(x_bf16, dtype=np.uint16))
    cols = x.shape[-1]
    assert cols % group == 0
    g = x.reshape(-1, cols // group, group)
    amax = np.max(np.abs(g), axis=-1)
    _, e = np.frexp(amax)  # amax = f * 2^e, f in [0.5, 1): floor(log2(amax)) = e - 1
    shared = np.where(amax > 0, e.astype(np.int64) - 1 - 8, 0)
    shared = np.clip(shared, -127, 127)
    y = (g / np.ldexp(np.float32(1.0), shared)[..., None].astype(np.float32)).astype(np.float32)
    codes = e4m3_encode_array(y).reshape(x.shape)
    scales = (shared + 127).astype(np.uint8).reshape(*x.shape[:-1], cols // group)
    return codes, scales


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """Bit-exact widening of bf16 bits to float32 (a shift; used for inspection and fixtures)."""
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bits, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)
