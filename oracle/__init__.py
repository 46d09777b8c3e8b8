"""CPU oracle for split-KV decode attention and FFD top-delta decode.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package; the product path never does.
It shares no code with the CUDA library: the arithmetic lives in
``fd_oracle.c`` (binary64 attention, binary32 key encoding), compiled with gcc
by ``oracle/build.py``.  This module only marshals numpy arrays.

Functions (each follows the passage cited in ``fd_oracle.c``):
  decode_dense        standard attention, "Flash Decoding" tutorial section 1
  decode_dense_f64    the same with binary64 K/V (for reductions)
  decode_split        per-chunk (m_i, l_i, O_i) + the section-2 merge
  decode_paged        page gather + the dense definition (tutorial section 3)
  quantize_keys       2-bit body + int8 residual encoding (FFD summary section 5)
  dequantize_keys     k~ = deq2 (+ deq8) as binary64
  decode_topdelta     FFD pipeline, Fig. 2 order (sections 3-5)
  decode_topdelta_group_union
                      the same selection rule per query head, the union of
                      the sets over the heads that share a KV head, attention
                      of every head of the group over that union
  float_to_half       IEEE binary32 -> binary16, round to nearest even
  quantize_kv_fp8     per-row scaled e4m3 KV cache encoding
  dequantize_kv_fp8   its exact binary64 values
  float_to_e4m3       binary32 -> e4m3 (RNE, saturating)
  quantize_kv_fp4     e2m1 codes with power-of-two scales per 32-channel block
  dequantize_kv_fp4   its exact binary64 values
  quantize_v_fp4      the same encoding in the value layout (two tokens per byte)
  dequantize_v_fp4    its exact binary64 values
  decode_dense_fp8/4  the dense definition over the decoded cache
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.library_path()
        if not os.path.exists(path) or _build.is_stale():
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_decode_dense.argtypes = [P, P, P, P, I, I, I, I, I, D, P, P, I]
        lib.oracle_decode_dense_f64.argtypes = [P, P, P, P, I, I, I, I, I, D, P, P, I]
        lib.oracle_decode_split.argtypes = [P, P, P, P, I, I, I, I, I, D, I, P, P, P, P, P, I]
        lib.oracle_decode_paged.argtypes = [P, P, P, P, I, I, P, I, I, I, I, I, D, P, P, I]
        lib.oracle_quantize_keys.argtypes = [P, P, I, I, I, I, P, P, P, P, I]
        lib.oracle_dequantize_keys.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
        lib.oracle_decode_topdelta.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, D, I, I,
                                               P, P, P, P, P, P, I]
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_max_threads.argtypes = []
        lib.oracle_float_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_quantize_kv_fp8.argtypes = [P, P, I, I, I, I, P, P, I]
        lib.oracle_dequantize_kv_fp8.argtypes = [P, P, P, I, I, I, I, P]
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_double_to_e2m1.argtypes = [ctypes.c_double]
        lib.oracle_double_to_e2m1.restype = ctypes.c_uint8
        lib.oracle_fp4_block_exponent.argtypes = [ctypes.c_double]
        lib.oracle_fp4_block_exponent.restype = ctypes.c_int
        lib.oracle_quantize_kv_fp4.argtypes = [P, P, I, I, I, I, P, P, I]
        lib.oracle_dequantize_kv_fp4.argtypes = [P, P, P, I, I, I, I, P]
        for name in ("oracle_decode_dense", "oracle_decode_dense_f64", "oracle_decode_split",
                     "oracle_decode_paged", "oracle_quantize_keys", "oracle_dequantize_keys",
                     "oracle_decode_topdelta", "oracle_max_threads", "oracle_quantize_kv_fp8",
                     "oracle_dequantize_kv_fp8", "oracle_quantize_kv_fp4", "oracle_dequantize_kv_fp4"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    """bf16 / fp16 bit patterns as a C-contiguous uint16 array.  Accepts numpy
    uint16 arrays or torch bfloat16/float16 CPU tensors."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().cpu().contiguous()
        if a.dtype in (torch.bfloat16, torch.float16):
            a = a.view(torch.int16)
        a = a.numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        if a.dtype == np.int16:
            a = a.view(np.uint16)
        else:
            raise TypeError(f"expected 16-bit bit patterns, got {a.dtype}")
    return a


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def decode_dense(q, k, v, seq_lens, scale, n_threads=0):
    """q [B,Hq,d], k/v [B,Hkv,L_max,d] (bf16 bits), seq_lens [B] or None.
    Returns (out [B,Hq,d] f64, lse [B,Hq] f64)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, d = q.shape
    _, Hkv, L_max, _ = k.shape
    sl = _i32(seq_lens)
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = _load().oracle_decode_dense(_ptr(q), _ptr(k), _ptr(v), _ptr(sl), B, Hq, Hkv, L_max, d,
                                     float(scale), _ptr(out), _ptr(lse), int(n_threads))
    _check(rc, "decode_dense")
    return out, lse


def decode_dense_f64(q, k, v, seq_lens, scale, n_threads=0):
    """Same as decode_dense with binary64 q, K, V."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    B, Hq, d = q.shape
    _, Hkv, L_max, _ = k.shape
    sl = _i32(seq_lens)
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = _load().oracle_decode_dense_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(sl), B, Hq, Hkv, L_max, d,
                                         float(scale), _ptr(out), _ptr(lse), int(n_threads))
    _check(rc, "decode_dense_f64")
    return out, lse


def decode_split(q, k, v, seq_lens, scale, num_splits, n_threads=0):
    """Split form.  Returns (out, lse, part_m [B,Hq,S], part_l [B,Hq,S], part_o [B,Hq,S,d])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, d = q.shape
    _, Hkv, L_max, _ = k.shape
    S = int(num_splits)
    sl = _i32(seq_lens)
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    pm = np.empty((B, Hq, S), np.float64)
    pl = np.empty((B, Hq, S), np.float64)
    po = np.empty((B, Hq, S, d), np.float64)
    rc = _load().oracle_decode_split(_ptr(q), _ptr(k), _ptr(v), _ptr(sl), B, Hq, Hkv, L_max, d,
                                     float(scale), S, _ptr(out), _ptr(lse), _ptr(pm), _ptr(pl),
                                     _ptr(po), int(n_threads))
    _check(rc, "decode_split")
    return out, lse, pm, pl, po


def decode_paged(q, k_pages, v_pages, page_table, num_pages, seq_lens, scale, n_threads=0):
    """k_pages/v_pages [P,Hkv,page_size,d] (bf16 bits), page_table [B,max_pages] int32."""
    q, kp, vp = _u16(q), _u16(k_pages), _u16(v_pages)
    B, Hq, d = q.shape
    _, Hkv, page_size, _ = kp.shape
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    max_pages = pt.shape[1]
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = _load().oracle_decode_paged(_ptr(q), _ptr(kp), _ptr(vp), _ptr(pt), max_pages,
                                     int(num_pages), _ptr(sl), page_size, B, Hq, Hkv, d,
                                     float(scale), _ptr(out), _ptr(lse), int(n_threads))
    _check(rc, "decode_paged")
    return out, lse


def quantize_keys(k, seq_lens=None, n_threads=0):
    """k [B,Hkv,L_max,d] bf16 bits.  Returns (codes u8 [B,Hkv,L_max,d/4],
    mn_scale u16 [B,Hkv,L_max,d/32,2], res i8 [B,Hkv,L_max,d], res_scale u16 [B,Hkv,L_max,d/32]).
    Rows past seq_lens[b] are zero (never written by the encoder)."""
    k = _u16(k)
    B, Hkv, L_max, d = k.shape
    sl = _i32(seq_lens)
    codes = np.zeros((B, Hkv, L_max, d // 4), np.uint8)
    ms = np.zeros((B, Hkv, L_max, d // 32, 2), np.uint16)
    res = np.zeros((B, Hkv, L_max, d), np.int8)
    rs = np.zeros((B, Hkv, L_max, d // 32), np.uint16)
    rc = _load().oracle_quantize_keys(_ptr(k), _ptr(sl), B, Hkv, L_max, d, _ptr(codes), _ptr(ms),
                                      _ptr(res), _ptr(rs), int(n_threads))
    _check(rc, "quantize_keys")
    return codes, ms, res, rs


def dequantize_keys(codes, mn_scale, res, res_scale, seq_lens=None, with_residual=True):
    codes = np.ascontiguousarray(codes, np.uint8)
    ms = np.ascontiguousarray(mn_scale, np.uint16)
    res = np.ascontiguousarray(res, np.int8)
    rs = np.ascontiguousarray(res_scale, np.uint16)
    B, Hkv, L_max, d4 = codes.shape
    d = d4 * 4
    sl = _i32(seq_lens)
    kt = np.empty((B, Hkv, L_max, d), np.float64)
    rc = _load().oracle_dequantize_keys(_ptr(codes), _ptr(ms), _ptr(res), _ptr(rs), _ptr(sl), B, Hkv,
                                        L_max, d, int(bool(with_residual)), _ptr(kt))
    _check(rc, "dequantize_keys")
    return kt


def decode_topdelta(q, codes, mn_scale, res, res_scale, v, seq_lens, scale, delta,
                    n_sink=4, window=64, want_scores=False, n_threads=0):
    """Returns a dict with out [B,Hq,d], lse [B,Hq], sel_mask [B,Hq,ceil(L/32)] u32,
    sel_count [B,Hq], m_hat [B,Hq] and (optionally) s_tilde [B,Hq,L_max]."""
    q, v = _u16(q), _u16(v)
    codes = np.ascontiguousarray(codes, np.uint8)
    ms = np.ascontiguousarray(mn_scale, np.uint16)
    res = np.ascontiguousarray(res, np.int8)
    rs = np.ascontiguousarray(res_scale, np.uint16)
    B, Hq, d = q.shape
    _, Hkv, L_max, _ = v.shape
    sl = _i32(seq_lens)
    words = (L_max + 31) // 32
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    mask = np.zeros((B, Hq, words), np.uint32)
    cnt = np.zeros((B, Hq), np.int32)
    mh = np.empty((B, Hq), np.float64)
    st = np.full((B, Hq, L_max), np.nan, np.float64) if want_scores else None
    dl = math.inf if delta is None else float(delta)
    rc = _load().oracle_decode_topdelta(_ptr(q), _ptr(codes), _ptr(ms), _ptr(res), _ptr(rs), _ptr(v),
                                        _ptr(sl), B, Hq, Hkv, L_max, d, float(scale), dl,
                                        int(n_sink), int(window), _ptr(out), _ptr(lse), _ptr(mask),
                                        _ptr(cnt), _ptr(mh), _ptr(st), int(n_threads))
    _check(rc, "decode_topdelta")
    r = dict(out=out, lse=lse, sel_mask=mask, sel_count=cnt, m_hat=mh)
    if want_scores:
        r["s_tilde"] = st
    return r


def float_to_half(x) -> np.ndarray:
    """Element-wise IEEE binary32 -> binary16 bits (round to nearest even)."""
    lib = _load()
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib.oracle_float_to_half(float(v)) for v in x], np.uint16)


def half_to_float(h) -> np.ndarray:
    lib = _load()
    h = np.asarray(h, np.uint16).ravel()
    return np.array([lib.oracle_half_to_float(int(v)) for v in h], np.float32)


def float_to_e4m3(x) -> np.ndarray:
    """Element-wise binary32 -> e4m3 code (round to nearest even, saturating at 448)."""
    lib = _load()
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib.oracle_float_to_e4m3(float(v)) for v in x], np.uint8)


def e4m3_value(c) -> np.ndarray:
    lib = _load()
    c = np.asarray(c, np.uint8).ravel()
    return np.array([lib.oracle_e4m3_value(int(v)) for v in c], np.float64)


def quantize_kv_fp8(x, seq_lens=None, n_threads=0):
    """x [B,H,L_max,d] bf16 bits -> (codes u8 [B,H,L_max,d], scales f32 [B,H,L_max]);
    rows past seq_lens[b] are zero."""
    x = _u16(x)
    B, H, L_max, d = x.shape
    sl = _i32(seq_lens)
    codes = np.zeros((B, H, L_max, d), np.uint8)
    scales = np.zeros((B, H, L_max), np.float32)
    rc = _load().oracle_quantize_kv_fp8(_ptr(x), _ptr(sl), B, H, L_max, d, _ptr(codes), _ptr(scales),
                                        int(n_threads))
    _check(rc, "quantize_kv_fp8")
    return codes, scales


def dequantize_kv_fp8(codes, scales, seq_lens=None):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    B, H, L_max, d = codes.shape
    sl = _i32(seq_lens)
    out = np.empty((B, H, L_max, d), np.float64)
    rc = _load().oracle_dequantize_kv_fp8(_ptr(codes), _ptr(scales), _ptr(sl), B, H, L_max, d, _ptr(out))
    _check(rc, "dequantize_kv_fp8")
    return out


def decode_dense_fp8(q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, n_threads=0):
    """Attention over an fp8 cache: the dense definition (tutorial section 1)
    evaluated in binary64 on the dequantized K~ = e4m3(code) * s rows.
    q [B,Hq,d] bf16 bits; codes [B,Hkv,L_max,d] u8; scales [B,Hkv,L_max] f32."""
    q = _u16(q)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kt = dequantize_kv_fp8(k_codes, k_scales, seq_lens)
    vt = dequantize_kv_fp8(v_codes, v_scales, seq_lens)
    return decode_dense_f64(qf, kt, vt, seq_lens, scale, n_threads)


def e2m1_value(c) -> np.ndarray:
    lib = _load()
    c = np.asarray(c, np.uint8).ravel()
    return np.array([lib.oracle_e2m1_value(int(v)) for v in c], np.float64)


def to_e2m1(y) -> np.ndarray:
    """Element-wise nearest e2m1 code (ties to even, saturating at 6)."""
    lib = _load()
    y = np.asarray(y, np.float64).ravel()
    return np.array([lib.oracle_double_to_e2m1(float(v)) for v in y], np.uint8)


def fp4_block_exponent(amax) -> int:
    return int(_load().oracle_fp4_block_exponent(float(amax)))


def quantize_kv_fp4(x, seq_lens=None, n_threads=0):
    """x [B,H,L_max,d] bf16 bits -> (codes u8 [B,H,L_max,d/2], scales u8 [B,H,L_max,d/32]);
    rows past seq_lens[b] are zero."""
    x = _u16(x)
    B, H, L_max, d = x.shape
    sl = _i32(seq_lens)
    codes = np.zeros((B, H, L_max, d // 2), np.uint8)
    scales = np.zeros((B, H, L_max, d // 32), np.uint8)
    rc = _load().oracle_quantize_kv_fp4(_ptr(x), _ptr(sl), B, H, L_max, d, _ptr(codes), _ptr(scales),
                                        int(n_threads))
    _check(rc, "quantize_kv_fp4")
    return codes, scales


def dequantize_kv_fp4(codes, scales, seq_lens=None):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    B, H, L_max, d2 = codes.shape
    d = 2 * d2
    sl = _i32(seq_lens)
    out = np.empty((B, H, L_max, d), np.float64)
    rc = _load().oracle_dequantize_kv_fp4(_ptr(codes), _ptr(scales), _ptr(sl), B, H, L_max, d, _ptr(out))
    _check(rc, "dequantize_kv_fp4")
    return out


def fp4_rows_to_pairs(codes, seq_lens=None):
    """Re-lay fp4 codes stored two channels per byte ([B,H,L,d/2], the key
    layout) into the value layout, two tokens per byte ([B,H,(L+1)/2,d]):
    byte (p, c) = code(2p+1, c) << 4 | code(2p, c).  A token at or past
    seq_lens[b] contributes code 0; a pair whose first token is past it stays
    zero.  Pure data movement (nibbles), no arithmetic."""
    codes = np.ascontiguousarray(codes, np.uint8)
    B, H, L, d2 = codes.shape
    d = 2 * d2
    nib = np.empty((B, H, L + (L % 2), d), np.uint8)
    nib[:, :, :L, 0::2] = codes & 0x0F
    nib[:, :, :L, 1::2] = codes >> 4
    if L % 2:
        nib[:, :, L] = 0
    lens = [L] * B if seq_lens is None else [int(x) for x in _i32(seq_lens)]
    for b, Lb in enumerate(lens):
        nib[b, :, Lb:] = 0
    pairs = (nib[:, :, 1::2] << 4) | nib[:, :, 0::2]
    for b, Lb in enumerate(lens):
        pairs[b, :, (Lb + 1) // 2:] = 0
    return np.ascontiguousarray(pairs, np.uint8)


def fp4_pairs_to_rows(pairs, L):
    """Inverse of fp4_rows_to_pairs for the first L tokens: [B,H,(L+1)/2,d]
    -> [B,H,L,d/2] (two channels per byte)."""
    pairs = np.ascontiguousarray(pairs, np.uint8)
    B, H, P, d = pairs.shape
    nib = np.empty((B, H, 2 * P, d), np.uint8)
    nib[:, :, 0::2] = pairs & 0x0F
    nib[:, :, 1::2] = pairs >> 4
    nib = nib[:, :, :L]
    return np.ascontiguousarray((nib[..., 1::2] << 4) | nib[..., 0::2], np.uint8)


def quantize_v_fp4(x, seq_lens=None, n_threads=0):
    """The fp4 encoding of quantize_kv_fp4 in the value layout: (codes u8
    [B,H,(L_max+1)/2,d] in token pairs, scales u8 [B,H,L_max,d/32])."""
    codes, scales = quantize_kv_fp4(x, seq_lens, n_threads)
    return fp4_rows_to_pairs(codes, seq_lens), scales


def dequantize_v_fp4(pairs, scales, seq_lens=None):
    """Decoded values of a token-pair fp4 value cache (binary64 [B,H,L_max,d])."""
    scales = np.ascontiguousarray(scales, np.uint8)
    return dequantize_kv_fp4(fp4_pairs_to_rows(pairs, scales.shape[2]), scales, seq_lens)


def decode_dense_fp4(q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, n_threads=0):
    """Attention over an fp4 cache: the dense definition (tutorial section 1)
    in binary64 on the decoded rows e2m1(code) * 2^e of K (key layout) and V
    (token-pair value layout)."""
    q = _u16(q)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kt = dequantize_kv_fp4(k_codes, k_scales, seq_lens)
    vt = dequantize_v_fp4(v_codes, v_scales, seq_lens)
    return decode_dense_f64(qf, kt, vt, seq_lens, scale, n_threads)


def _bf16_to_f64(a):
    """bf16 bit patterns (uint16) -> their exact binary64 values."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_topdelta_group_union(q, codes, mn_scale, res, res_scale, v, seq_lens, scale, delta,
                                n_sink=4, window=64, want_scores=False, n_threads=0):
    """Top-delta with one candidate set per KV group (FFD summary: the rule
    of section 3 and the pseudo-max of section 4 per query head, Fig. 2's
    exact attention over the candidates; the set shared by a group is this
    library's option, not the page's).  Steps:
      1-3. Sel_g per query head g, exactly as decode_topdelta;
      4.   Sel_group = union of Sel_g over the G heads that read one KV head;
      5.   every head of the group: softmax over Sel_group of the residual-
           corrected scores s_j = scale * <q, k~_j> (k~ from dequantize_keys),
           times the bf16 V rows -- the binary64 dense definition
           (decode_dense_f64) restricted to the tokens of Sel_group.
    Returns decode_topdelta's dict with sel_mask / sel_count describing the
    attended set (Sel_group, the same for every head of a group), plus
    head_sel_mask / head_sel_count (each head's own Sel_g) and m_hat."""
    per_head = decode_topdelta(q, codes, mn_scale, res, res_scale, v, seq_lens, scale, delta, n_sink, window,
                               want_scores=want_scores, n_threads=n_threads)
    q, v = _u16(q), _u16(v)
    B, Hq, d = q.shape
    _, Hkv, L_max, _ = v.shape
    G = Hq // Hkv
    words = per_head["sel_mask"].shape[-1]
    group = np.bitwise_or.reduce(per_head["sel_mask"].reshape(B, Hkv, G, words), axis=2)     # [B, Hkv, words]
    sel = np.unpackbits(group.view(np.uint8), axis=-1, bitorder="little")[..., :L_max].astype(bool)
    kt = dequantize_keys(codes, mn_scale, res, res_scale, seq_lens)
    qf, vf = _bf16_to_f64(q), _bf16_to_f64(v)
    lens = [L_max] * B if seq_lens is None else [int(x) for x in _i32(seq_lens)]
    out = np.zeros((B, Hq, d), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    cnt = np.zeros((B, Hq), np.int32)
    for b in range(B):
        for h in range(Hkv):
            idx = np.nonzero(sel[b, h, :lens[b]])[0]
            cnt[b, h * G:(h + 1) * G] = idx.size
            if idx.size == 0:
                continue
            o, l = decode_dense_f64(qf[b:b + 1, h * G:(h + 1) * G], kt[b:b + 1, h:h + 1, idx],
                                    vf[b:b + 1, h:h + 1, idx], None, scale, n_threads)
            out[b, h * G:(h + 1) * G] = o[0]
            lse[b, h * G:(h + 1) * G] = l[0]
    r = dict(out=out, lse=lse, sel_mask=np.repeat(group, G, axis=1), sel_count=cnt, m_hat=per_head["m_hat"],
             head_sel_mask=per_head["sel_mask"], head_sel_count=per_head["sel_count"])
    if want_scores:
        r["s_tilde"] = per_head["s_tilde"]
    return r
