"""CPU oracle for FP8-quantised paged decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The product library never imports, links or calls anything here,
and nothing here calls the product library.

The arithmetic lives in ``fp8pa_oracle.c`` (plain C, FP64 attention, FP8 by
explicit bit fields); this module only compiles it with gcc and marshals
numpy arrays into it.  Sources are cited in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2, INT8 = 0, 1, 2  # INT8: the symmetric alternate codec (FMAX 127)
SCALE_TOKEN_HEAD, SCALE_CHANNEL_STATIC, SCALE_TOKEN_GROUP, SCALE_MX_BLOCK = 0, 1, 2, 3
SCALE_SEGMENT = 4
SEGMENT_TOKENS = 1024

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i, d, L = ctypes.c_int, ctypes.c_double, ctypes.c_long
    lib.or_fp8_decode.argtypes = [ctypes.c_uint8, i]
    lib.or_fp8_decode.restype = d
    lib.or_fp8_encode.argtypes = [ctypes.c_float, i]
    lib.or_fp8_encode.restype = ctypes.c_uint8
    lib.or_fp8_encode_array.argtypes = [P, L, i, P]
    lib.or_fp8_encode_bruteforce_array.argtypes = [P, L, i, P]
    lib.or_fp8_decode_array.argtypes = [P, L, i, P]
    lib.or_absmax_scale_bf16.argtypes = [P, i, i]
    lib.or_absmax_scale_bf16.restype = ctypes.c_float
    lib.or_mx_exponent.argtypes = [ctypes.c_float, i]
    lib.or_mx_exponent.restype = i
    lib.or_kv_append_quant.argtypes = [P, P, P, i, i, i, i, i, i, P, P, P, P, i, i]
    lib.or_kv_append_quant.restype = i
    lib.or_kv_channel_scales.argtypes = [P, i, i, i, i, P]
    lib.or_kv_append_quant_segment.argtypes = [P, P, P, P, P, i, i, i, i, P, P, P, P, P, i, i]
    lib.or_kv_append_quant_segment.restype = i
    lib.or_paged_decode_attention.argtypes = [P, P, P, P, P, P, i, P, i, i, i, i, i, i, i, i, i,
                                              d, i, P, i, P, i]
    lib.or_paged_decode_attention.restype = i
    lib.or_attention_weights.argtypes = [P, P, P, P, i, P, i, i, i, i, i, i, i, d, i, i, i, P]
    lib.or_attention_weights.restype = i
    lib.or_attention_split_merge.argtypes = [P, P, P, P, P, P, i, P, i, i, i, i, i, i, i, i, i,
                                             d, i, i, P]
    lib.or_max_threads.restype = i
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().or_max_threads())


def fp8_decode(codes, fmt: int) -> np.ndarray:
    c = _c(np.asarray(codes), np.uint8).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    _load().or_fp8_decode_array(_ptr(c), c.size, fmt, _ptr(out))
    return out.reshape(np.shape(codes))


def fp8_encode(x, fmt: int) -> np.ndarray:
    a = _c(np.asarray(x), np.float32).reshape(-1)
    out = np.empty(a.size, dtype=np.uint8)
    _load().or_fp8_encode_array(_ptr(a), a.size, fmt, _ptr(out))
    return out.reshape(np.shape(x))


def fp8_encode_bruteforce(x, fmt: int) -> np.ndarray:
    a = _c(np.asarray(x), np.float32).reshape(-1)
    out = np.empty(a.size, dtype=np.uint8)
    _load().or_fp8_encode_bruteforce_array(_ptr(a), a.size, fmt, _ptr(out))
    return out.reshape(np.shape(x))


def mx_exponent(amax: float, fmt: int) -> int:
    """The MX block exponent e (scale 2^e) for a block absmax."""
    return int(_load().or_mx_exponent(ctypes.c_float(amax), fmt))


def absmax_scale(x_bf16, fmt: int) -> float:
    a = _c(np.asarray(x_bf16), np.uint16).reshape(-1)
    return float(_load().or_absmax_scale_bf16(_ptr(a), a.size, fmt))


def kv_append_quant(k, v, slot_mapping, fmt, scale_mode, group_size, k_cache, v_cache,
                    k_scale, v_scale, block_size) -> int:
    """In-place append into numpy caches; k/v are bf16 bit patterns (uint16)
    of shape [num_tokens, Hkv, D].  Returns the count of out-of-range slots."""
    if fmt == INT8 and scale_mode == SCALE_MX_BLOCK:
        raise ValueError("the power-of-two block mode is defined for FP8 codes only")
    if scale_mode == SCALE_SEGMENT:
        raise ValueError("the segment mode needs positions: use kv_append_quant_segment")
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    sdt = np.uint8 if scale_mode == SCALE_MX_BLOCK else np.float32  # E8M0 bytes
    for arr, dt in ((k_cache, np.uint8), (k_scale, sdt)):
        assert arr.dtype == dt and arr.flags.c_contiguous
    if v is not None:
        assert v_cache.dtype == np.uint8 and v_cache.flags.c_contiguous
        assert v_scale.dtype == sdt and v_scale.flags.c_contiguous
    n, hkv, d = k.shape
    num_blocks = k_cache.shape[0]
    return int(_load().or_kv_append_quant(_ptr(k), _ptr(v), _ptr(sm), n, hkv, d, fmt, scale_mode,
                                          group_size, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                          _ptr(v_scale), num_blocks, block_size))


def segment_scale_heads(n_kv_heads: int) -> int:
    """Row length of the segment scale array: KV heads rounded up to 4."""
    return (n_kv_heads + 3) // 4 * 4


def kv_append_quant_segment(k, v, slot_mapping, seq_offsets, seq_start_pos, fmt, seg_state,
                            k_cache, v_cache, k_scale, v_scale, block_size) -> int:
    """Segment-scale append (block-wise cumulative rescaling), in place.
    k/v: bf16 bits [num_tokens, Hkv, D]; sequence r owns rows
    seq_offsets[r]:seq_offsets[r+1] at positions seq_start_pos[r] + 0, 1, ...;
    seg_state: float32 [num_seqs, 2, Hkv, 2] (running absmax, segment scale),
    updated; scales: float32 [num_blocks, round_up(Hkv, 4)].  Returns the
    count of out-of-range slots."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    off = _c(seq_offsets, np.int32)
    sp = _c(seq_start_pos, np.int32)
    n, hkv, d = k.shape
    assert off.size == sp.size + 1 and int(off[-1]) <= n
    assert seg_state.dtype == np.float32 and seg_state.flags.c_contiguous
    assert seg_state.shape == (sp.size, 2, hkv, 2)
    hp = segment_scale_heads(hkv)
    for arr in (k_scale, v_scale):
        if arr is not None:
            assert arr.dtype == np.float32 and arr.flags.c_contiguous
            assert arr.shape == (k_cache.shape[0], hp)
    return int(_load().or_kv_append_quant_segment(
        _ptr(k), _ptr(v), _ptr(sm), _ptr(off), _ptr(sp), sp.size, hkv, d, fmt, _ptr(seg_state),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), k_cache.shape[0],
        block_size))


def kv_channel_scales(x, fmt: int) -> np.ndarray:
    x = _c(x, np.uint16)
    n, hkv, d = x.shape
    out = np.empty((hkv, d), dtype=np.float32)
    _load().or_kv_channel_scales(_ptr(x), n, hkv, d, fmt, _ptr(out))
    return out


def paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                           block_size, n_kv_heads, head_dim_v, fmt, scale_mode, group_size,
                           sm_scale, rows=None, num_threads=None):
    """FP64 attention over the paged cache.  q: bf16 bits [B, Hq, Dk].
    Returns float64 [B, Hq, Dv] (rows=None) or [len(rows), Dv]."""
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, hq, dk = q.shape
    if rows is not None:
        rows = _c(rows, np.int32)
        out = np.zeros((rows.size, head_dim_v), dtype=np.float64)
    else:
        out = np.zeros((B, hq, head_dim_v), dtype=np.float64)
    nt = num_threads or max_threads()
    bad = _load().or_paged_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(bt),
        bt.shape[1], _ptr(sl), B, block_size, hq, n_kv_heads, dk, head_dim_v, fmt, scale_mode,
        group_size, float(sm_scale), k_cache.shape[0], _ptr(rows),
        0 if rows is None else rows.size, _ptr(out), nt)
    if bad:
        raise ValueError(f"oracle: {bad} rows read an out-of-range block id")
    return out


def attention_weights(q, k_cache, k_scale, block_tables, seq_lens, block_size, n_kv_heads, fmt,
                      scale_mode, group_size, sm_scale, b, h):
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, hq, dk = q.shape
    w = np.zeros(int(bt.shape[1] * block_size) + 1, dtype=np.float64)
    n = _load().or_attention_weights(_ptr(q), _ptr(k_cache), _ptr(k_scale), _ptr(bt), bt.shape[1],
                                     _ptr(sl), block_size, hq, n_kv_heads, dk, fmt, scale_mode,
                                     group_size, float(sm_scale), k_cache.shape[0], b, h, _ptr(w))
    return w[:n]


def attention_split_merge(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                          block_size, n_kv_heads, head_dim_v, fmt, scale_mode, group_size,
                          sm_scale, chunk_tokens):
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, hq, dk = q.shape
    out = np.zeros((B, hq, head_dim_v), dtype=np.float64)
    _load().or_attention_split_merge(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(bt), bt.shape[1], _ptr(sl), B, block_size,
                                     hq, n_kv_heads, dk, head_dim_v, fmt, scale_mode, group_size,
                                     float(sm_scale), k_cache.shape[0], int(chunk_tokens),
                                     _ptr(out))
    return out


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
