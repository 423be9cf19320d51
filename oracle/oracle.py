"""ctypes wrapper of the CPU oracle (kvq_oracle.c).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and the CPU legs of
bench.py import this module.  It shares no code with the CUDA library
(bit_kv_cache_keyquant_gb300) and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden", "-Wall", "-Wno-unused-function"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no CUDA) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


P = ctypes.c_void_p
I = ctypes.c_int
L = ctypes.c_long
D = ctypes.c_double
U16 = ctypes.c_uint16
U64 = ctypes.c_uint64
I32 = ctypes.c_int32


def _declare(l):
    sig = {
        "orc_half_to_double": (D, [U16]),
        "orc_double_to_half": (U16, [D, I]),
        "orc_affine_fit": (None, [P, L, L, I, P, P]),
        "orc_affine_code": (I, [U16, U16, U16, I]),
        "orc_affine_dequant": (D, [I, U16, U16]),
        "orc_kivi_key_codes": (None, [I, I, I, P, L, P, P]),
        "orc_kivi_key_byte_offset": (L, [I, I]),
        "orc_kivi_key_bit": (I, [I]),
        "orc_kivi_key_pack": (I, [I, I, P, L, P]),
        "orc_kivi_key_byte_offset_w": (L, [I, I, I]),
        "orc_kivi_key_bit_w": (I, [I, I]),
        "orc_kivi_key_pack_w": (I, [I, I, I, P, L, P]),
        "orc_tokenmajor_pack_w": (None, [I, I, P, L, P]),
        "orc_kivi_value_byte_offset": (L, [I, I]),
        "orc_kivi_value_bit": (I, [I]),
        "orc_kivi_value_byte_offset4": (L, [I, I]),
        "orc_kivi_value_bit4": (I, [I]),
        "orc_kivi_value_pack_w": (I, [I, I, I, P, L, P]),
        "orc_kivi_decode_one_w": (None, [I, I, I, I, I, I, I, I, I, D, P, P, P, P, P, P, P, P]),
        "orc_kivi_key_sz_index": (I, [I]),
        "orc_kivi_key_sz_pack": (I, [I, P, L, P]),
        "orc_kivi_value_codes": (None, [I, I, I, P, L, P, P]),
        "orc_tokenmajor_pack": (None, [I, P, L, P]),
        "orc_kitty_key_page_bytes": (L, [I, I, I]),
        "orc_kitty_high_rows": (I, [I]),
        "orc_kitty_low_byte_offset": (L, [I, I]),
        "orc_kitty_high_byte_offset": (L, [I, I, I]),
        "orc_kitty_code_bit": (I, [I]),
        "orc_kitty_value_page_bytes": (L, [I, I]),
        "orc_kitty_select": (None, [I, I, I, I, P, P]),
        "orc_kitty_key_page": (None, [I, I, I, I, P, P]),
        "orc_kitty_key_page_decode": (None, [I, I, I, P, P, P, P]),
        "orc_kitty_value_page": (None, [I, I, P, P]),
        "orc_philox4x32_10": (None, [P, P, P]),
        "orc_philox4x32_10_inverse": (None, [P, P, P]),
        "orc_dither": (ctypes.c_float, [U64, I32, I32, I, I32, I32, I32]),
        "orc_int8_quant_block": (None, [I, I, P, U64, I32, I32, I, I32, I32, P, P]),
        "orc_int8_dequant": (D, [I, U16, ctypes.c_float]),
        "orc_attend_fp16": (None, [I, I, P, P, P, D, P]),
        "orc_kivi_decode_one": (None, [I, I, I, I, I, I, D, P, P, P, P, P, P, P, P]),
        "orc_kitty_decode_one": (None, [I, I, I, I, I, I, I, D, P, P, P, P, P, P, P, P, P]),
        "orc_int8_decode_one": (None, [I, I, I, I, D, U64, I32, I32, I32, P, P, P, P, P, P, P, P]),
        "orc_dither_slot": (ctypes.c_float, [U64, I32, I, I32, I32, I32]),
        "orc_int8t_quant_token": (None, [I, I, P, U64, I32, I, I32, I32, P, P]),
        "orc_int8t_decode_one": (None, [I, I, I, I, I, D, U64, I32, I32, P, P, P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(l, name)
        f.restype = res
        f.argtypes = args


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _h16(a) -> np.ndarray:
    """View an fp16 array as its uint16 bit patterns (contiguous)."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint16) if a.dtype == np.float16 else a.astype(np.uint16)


# ---------------------------------------------------------------------------
# scalar helpers
# ---------------------------------------------------------------------------
RN, RD, RU = 0, 1, 2


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(bits)


def double_to_half(x: float, mode: int = RN) -> int:
    return lib().orc_double_to_half(x, mode)


def affine_fit(x_fp16: np.ndarray, bits: int):
    x = _h16(x_fp16).ravel()
    s, z = U16(), U16()
    lib().orc_affine_fit(_p(x), x.size, 1, bits, ctypes.byref(s), ctypes.byref(z))
    return s.value, z.value


def affine_code(x_bits: int, s: int, z: int, bits: int) -> int:
    return lib().orc_affine_code(x_bits, s, z, bits)


# ---------------------------------------------------------------------------
# KIVI
# ---------------------------------------------------------------------------
def kivi_key_codes(x: np.ndarray, bits: int = 2):
    """x fp16 [n_grp][G][D] -> (codes uint8 [n_grp][G][D], sz uint16 [n_grp][D][2])."""
    n, G, Dm = x.shape
    xb = _h16(x)
    codes = np.zeros((n, G, Dm), np.uint8)
    sz = np.zeros((n, Dm, 2), np.uint16)
    lib().orc_kivi_key_codes(Dm, G, bits, _p(xb), n, _p(codes), _p(sz))
    return codes, sz


def kivi_key_pack(codes: np.ndarray, bits: int = 2) -> np.ndarray:
    n, G, Dm = codes.shape
    out = np.zeros((n, G * Dm * bits // 8), np.uint8)
    rc = lib().orc_kivi_key_pack_w(Dm, G, bits, _p(np.ascontiguousarray(codes)), n, _p(out))
    if rc:
        raise ValueError("KIVI key packing needs D == 128, G % 32 == 0 and 2 or 4 bits")
    return out


def kivi_key_byte_offset(t: int, c: int, bits: int = 2) -> int:
    return lib().orc_kivi_key_byte_offset_w(bits, t, c)


def kivi_key_bit(t: int, bits: int = 2) -> int:
    return lib().orc_kivi_key_bit_w(bits, t)


def kivi_key_sz_index(c: int) -> int:
    return lib().orc_kivi_key_sz_index(c)


def kivi_key_sz_pack(sz: np.ndarray) -> np.ndarray:
    """sz uint16 [n_grp][D][2] (scale, zero) -> stored blocks uint16 [n_grp][2*D]."""
    n, Dm, _ = sz.shape
    out = np.zeros((n, 2 * Dm), np.uint16)
    if lib().orc_kivi_key_sz_pack(Dm, _p(np.ascontiguousarray(sz)), n, _p(out)):
        raise ValueError("KIVI key parameter packing needs D == 128")
    return out


def kivi_quant_key(x: np.ndarray, bits: int = 2):
    """Full a1 step: fp16 [n_grp][G][D] -> (packed codes, sz)."""
    codes, sz = kivi_key_codes(x, bits)
    return kivi_key_pack(codes, bits), sz


def kivi_value_codes(x: np.ndarray, group: int = 32, bits: int = 2):
    n, Dm = x.shape
    xb = _h16(x)
    codes = np.zeros((n, Dm), np.uint8)
    sz = np.zeros((n, Dm // group, 2), np.uint16)
    lib().orc_kivi_value_codes(Dm, group, bits, _p(xb), n, _p(codes), _p(sz))
    return codes, sz


def tokenmajor_pack(codes: np.ndarray, bits: int = 2) -> np.ndarray:
    n, Dm = codes.shape
    out = np.zeros((n, Dm * bits // 8), np.uint8)
    lib().orc_tokenmajor_pack_w(Dm, bits, _p(np.ascontiguousarray(codes)), n, _p(out))
    return out


def kivi_value_byte_offset(t: int, c: int) -> int:
    return lib().orc_kivi_value_byte_offset(t, c)


def kivi_value_bit(c: int) -> int:
    return lib().orc_kivi_value_bit(c)


def kivi_value_byte_offset4(t: int, c: int) -> int:
    return lib().orc_kivi_value_byte_offset4(t, c)


def kivi_value_bit4(c: int) -> int:
    return lib().orc_kivi_value_bit4(c)


def kivi_value_pack(codes: np.ndarray, bits: int = 2, tiles: bool = False) -> np.ndarray:
    """Value codes [n][D] -> the stored bytes as rows of D*bits/8: token-major (one row per token), or with
    tiles ceil(n/32) 32-token value tiles (32 rows each, in the tile order)."""
    n, Dm = codes.shape
    rows = (n + 31) // 32 * 32 if tiles else n
    out = np.zeros((rows, Dm * bits // 8), np.uint8)
    if lib().orc_kivi_value_pack_w(Dm, bits, int(tiles), _p(np.ascontiguousarray(codes)), n, _p(out)):
        raise ValueError("KIVI value packing needs D == 128 and 2 or 4 bits")
    return out


def kivi_quant_value(x: np.ndarray, group: int = 32, bits: int = 2, tiles: bool = False):
    codes, sz = kivi_value_codes(x, group, bits)
    return kivi_value_pack(codes, bits, tiles), sz


# ---------------------------------------------------------------------------
# Kitty
# ---------------------------------------------------------------------------
def kitty_key_page_bytes(D: int, G: int, K: int) -> int:
    return lib().orc_kitty_key_page_bytes(D, G, K)


def kitty_high_rows(K: int) -> int:
    return lib().orc_kitty_high_rows(K)


def kitty_low_byte_offset(t: int, c: int) -> int:
    return lib().orc_kitty_low_byte_offset(t, c)


def kitty_high_byte_offset(K: int, t: int, rho: int) -> int:
    return lib().orc_kitty_high_byte_offset(K, t, rho)


def kitty_code_bit(t: int) -> int:
    return lib().orc_kitty_code_bit(t)


def kitty_value_page_bytes(D: int, G: int) -> int:
    return lib().orc_kitty_value_page_bytes(D, G)


def kitty_select(x: np.ndarray, K: int, score_mode: int = 0) -> np.ndarray:
    G, Dm = x.shape
    out = np.zeros(Dm, np.uint8)
    lib().orc_kitty_select(Dm, G, K, score_mode, _p(_h16(x)), _p(out))
    return out


def kitty_key_page(x: np.ndarray, K: int, score_mode: int = 0) -> np.ndarray:
    G, Dm = x.shape
    out = np.zeros(kitty_key_page_bytes(Dm, G, K), np.uint8)
    lib().orc_kitty_key_page(Dm, G, K, score_mode, _p(_h16(x)), _p(out))
    return out


def kitty_key_page_decode(page: np.ndarray, D: int, G: int, K: int):
    codes = np.zeros((G, D), np.uint8)
    s = np.zeros(D, np.uint16)
    z = np.zeros(D, np.uint16)
    lib().orc_kitty_key_page_decode(D, G, K, _p(np.ascontiguousarray(page)), _p(codes), _p(s), _p(z))
    return codes, s, z


def kitty_value_page(x: np.ndarray) -> np.ndarray:
    G, Dm = x.shape
    out = np.zeros(kitty_value_page_bytes(Dm, G), np.uint8)
    lib().orc_kitty_value_page(Dm, G, _p(_h16(x)), _p(out))
    return out


# ---------------------------------------------------------------------------
# Philox / INT8 dither
# ---------------------------------------------------------------------------
def philox(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def philox_inverse(out, key):
    o = np.ascontiguousarray(np.asarray(out, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    ctr = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10_inverse(_p(o), _p(k), _p(ctr))
    return ctr


def dither(seed: int, request: int, layer: int, kv_sel: int, kv_head: int, token: int, channel: int) -> float:
    return lib().orc_dither(seed, request, layer, kv_sel, kv_head, token, channel)


def int8_quant_block(x: np.ndarray, seed: int, request: int, layer: int, kv_sel: int,
                     kv_head: int, tok0: int):
    T, Dm = x.shape
    codes = np.zeros((T, Dm), np.int8)
    scale = np.zeros(Dm, np.uint16)
    lib().orc_int8_quant_block(Dm, T, _p(_h16(x)), seed, request, layer, kv_sel, kv_head, tok0,
                               _p(codes), _p(scale))
    return codes, scale


def dither_slot(seed: int, layer: int, kv_sel: int, kv_head: int, slot: int, channel: int) -> float:
    return lib().orc_dither_slot(seed, layer, kv_sel, kv_head, slot, channel)


def int8t_quant_token(x: np.ndarray, Gc: int, seed: int, layer: int, kv_sel: int, kv_head: int, slot: int):
    """One token of one kv head written to `slot`: fp16 [D] -> (int8 codes [D], fp16 bits scales [D/Gc])."""
    Dm = x.shape[0]
    codes = np.zeros(Dm, np.int8)
    scale = np.zeros(Dm // Gc, np.uint16)
    lib().orc_int8t_quant_token(Dm, Gc, _p(_h16(x)), seed, layer, kv_sel, kv_head, slot, _p(codes), _p(scale))
    return codes, scale


def int8t_write(pool, K: np.ndarray, V: np.ndarray, slots, kv_head: int, Gc: int, seed: int, layer: int):
    """Quantize tokens K[i], V[i] ([n][D] fp16) of one kv head into pool slots slots[i].

    pool = (kc, vc, ks, vs): int8 [n_slots][Hkv][D] and uint16 [n_slots][Hkv][D/Gc], updated in place."""
    kc, vc, ks, vs = pool
    for i, s in enumerate(slots):
        kc[s, kv_head], ks[s, kv_head] = int8t_quant_token(K[i], Gc, seed, layer, 0, kv_head, int(s))
        vc[s, kv_head], vs[s, kv_head] = int8t_quant_token(V[i], Gc, seed, layer, 1, kv_head, int(s))


def int8t_decode_one(q, pool, table, kv_head: int, seed: int, layer: int, Gc: int = 32, sm_scale=None):
    """One (request, kv head) whose token t sits in slot table[t]: q fp16 [g][D] -> binary64 [g][D]."""
    kc, vc, ks, vs = pool
    g, Dm = q.shape
    Hkv = kc.shape[1]
    tab = np.ascontiguousarray(table, dtype=np.int32)
    sm = (1.0 / np.sqrt(Dm)) if sm_scale is None else sm_scale
    out = np.zeros((g, Dm), np.float64)
    lib().orc_int8t_decode_one(Dm, Gc, Hkv, len(tab), g, sm, seed, layer, kv_head, _p(tab), _p(_h16(q)),
                               _p(np.ascontiguousarray(kc)), _p(np.ascontiguousarray(vc)), _p(_h16(ks)),
                               _p(_h16(vs)), _p(out))
    return out


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def attend_fp16(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    n, Dm = k.shape
    out = np.zeros(Dm, np.float64)
    lib().orc_attend_fp16(Dm, n, _p(_h16(q)), _p(_h16(k)), _p(_h16(v)), sm_scale, _p(out))
    return out


def kivi_decode_one(q, kc, ksz, vc, vsz, kres, vres, L, G=32, Gv=32, R=128, sm_scale=None, bits_k=2, bits_v=2,
                    value_tiles=False):
    """One (batch row, kv head): q fp16 [g][D] -> binary64 [g][D]."""
    g, Dm = q.shape
    sm = (1.0 / np.sqrt(Dm)) if sm_scale is None else sm_scale
    out = np.zeros((g, Dm), np.float64)
    lib().orc_kivi_decode_one_w(Dm, G, Gv, R, L, bits_k, bits_v, int(value_tiles), g, sm, _p(_h16(q)), _p(np.ascontiguousarray(kc)),
                                _p(_h16(ksz)), _p(np.ascontiguousarray(vc)), _p(_h16(vsz)),
                                _p(_h16(kres)), _p(_h16(vres)), _p(out))
    return out


def kitty_decode_one(q, kp, vp, ksink, vsink, kqbuf, vqbuf, vlocal, L, G=128, K=16, S=32, R=128,
                     sm_scale=None):
    g, Dm = q.shape
    sm = (1.0 / np.sqrt(Dm)) if sm_scale is None else sm_scale
    out = np.zeros((g, Dm), np.float64)
    lib().orc_kitty_decode_one(Dm, G, K, S, R, L, g, sm, _p(_h16(q)), _p(np.ascontiguousarray(kp)),
                               _p(np.ascontiguousarray(vp)), _p(_h16(ksink)), _p(_h16(vsink)),
                               _p(_h16(kqbuf)), _p(_h16(vqbuf)), _p(_h16(vlocal)), _p(out))
    return out


def int8_decode_one(q, kc, vc, ks, vs, ktail, vtail, L, seed, request, layer, kv_head, T=256,
                    sm_scale=None):
    g, Dm = q.shape
    sm = (1.0 / np.sqrt(Dm)) if sm_scale is None else sm_scale
    out = np.zeros((g, Dm), np.float64)
    lib().orc_int8_decode_one(Dm, T, L, g, sm, seed, request, layer, kv_head, _p(_h16(q)),
                              _p(np.ascontiguousarray(kc)), _p(np.ascontiguousarray(vc)),
                              _p(_h16(ks)), _p(_h16(vs)), _p(_h16(ktail)), _p(_h16(vtail)), _p(out))
    return out


# ---------------------------------------------------------------------------
# cache state of one (batch row, kv head) at attention time, from fp16 K, V
# ---------------------------------------------------------------------------
def kivi_segments(L: int, R: int = 128):
    """(n_kq, n_vq): quantized key tokens (whole groups) and quantized values.

    KIVI section 3.3 with Kitty's insert -> attend -> quantize order: the key
    residual holds ((L-1) mod R) + 1 tokens, the value residual min(L, R)."""
    rk = ((L - 1) % R) + 1
    rv = min(L, R)
    return L - rk, L - rv


def kivi_build_one(K: np.ndarray, V: np.ndarray, G: int = 32, Gv: int = 32, R: int = 128, bits_k: int = 2,
                   bits_v: int = 2, value_tiles: bool = False):
    """fp16 K, V [L][D] -> (kc, ksz, vc, vsz, kres, vres) for one (b, kvh)."""
    L, Dm = K.shape
    nkq, nvq = kivi_segments(L, R)
    ng = nkq // G
    if ng:
        kc, ksz = kivi_quant_key(K[:ng * G].reshape(ng, G, Dm), bits_k)
    else:
        kc = np.zeros((0, G * Dm * bits_k // 8), np.uint8)
        ksz = np.zeros((0, Dm, 2), np.uint16)
    if nvq:
        vc, vsz = kivi_quant_value(V[:nvq], Gv, bits_v, value_tiles)
    else:
        vc = np.zeros((0, Dm * bits_v // 8), np.uint8)
        vsz = np.zeros((0, Dm // Gv, 2), np.uint16)
    kres = np.zeros((R, Dm), np.float16)
    vres = np.zeros((R, Dm), np.float16)
    for t in range(nkq, L):
        kres[t % R] = K[t]
    for t in range(nvq, L):
        vres[t % R] = V[t]
    return kc, ksz, vc, vsz, kres, vres


def kitty_segments(L: int, G: int = 128, S: int = 32, R: int = 128):
    """(n_key_pages, n_key_qbuf, n_value_pages, n_value_qbuf, n_local)."""
    nkb = ((L - S - 1) % G) + 1 if L > S else 0
    pk = (L - S - nkb) // G if L > S else 0
    E = max(0, L - S - R)
    nvb = ((E - 1) % G) + 1 if E > 0 else 0
    pv = (E - nvb) // G
    nloc = min(max(L - S, 0), R)
    return pk, nkb, pv, nvb, nloc


def kitty_build_one(K: np.ndarray, V: np.ndarray, G: int = 128, Kb: int = 16, S: int = 32,
                    R: int = 128, score_mode: int = 0):
    L, Dm = K.shape
    pk, nkb, pv, nvb, nloc = kitty_segments(L, G, S, R)
    kpb, vpb = kitty_key_page_bytes(Dm, G, Kb), kitty_value_page_bytes(Dm, G)
    kp = np.zeros((pk, kpb), np.uint8)
    vp = np.zeros((pv, vpb), np.uint8)
    for p in range(pk):
        kp[p] = kitty_key_page(K[S + p * G:S + (p + 1) * G], Kb, score_mode)
    for p in range(pv):
        vp[p] = kitty_value_page(V[S + p * G:S + (p + 1) * G])
    ksink = np.zeros((S, Dm), np.float16)
    vsink = np.zeros((S, Dm), np.float16)
    n_s = min(L, S)
    ksink[:n_s] = K[:n_s]
    vsink[:n_s] = V[:n_s]
    kq = np.zeros((G, Dm), np.float16)
    vq = np.zeros((G, Dm), np.float16)
    vl = np.zeros((R, Dm), np.float16)
    for t in range(S + pk * G, L):
        kq[(t - S) % G] = K[t]
    for t in range(S + pv * G, S + pv * G + nvb):
        vq[(t - S) % G] = V[t]
    for t in range(L - nloc, L):
        vl[t % R] = V[t]
    return kp, vp, ksink, vsink, kq, vq, vl


def int8_build_one(K: np.ndarray, V: np.ndarray, seed: int, request: int, layer: int,
                   kv_head: int, T: int = 256):
    L, Dm = K.shape
    ntail = ((L - 1) % T) + 1
    nq = L - ntail
    nb = nq // T
    kc = np.zeros((L, Dm), np.int8)
    vc = np.zeros((L, Dm), np.int8)
    ks = np.zeros((max(nb, 1), Dm), np.uint16)
    vs = np.zeros((max(nb, 1), Dm), np.uint16)
    for blk in range(nb):
        sl = slice(blk * T, (blk + 1) * T)
        kc[sl], ks[blk] = int8_quant_block(K[sl], seed, request, layer, 0, kv_head, blk * T)
        vc[sl], vs[blk] = int8_quant_block(V[sl], seed, request, layer, 1, kv_head, blk * T)
    kt = np.zeros((T, Dm), np.float16)
    vt = np.zeros((T, Dm), np.float16)
    for t in range(nq, L):
        kt[t % T] = K[t]
        vt[t % T] = V[t]
    return kc, vc, ks, vs, kt, vt
