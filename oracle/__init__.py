"""fp64 CPU oracle for paged GQA decode, block scoring, tiering, selection,
gather and identity-keyed re-admission.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (it never imports it, nor its header) and reads its inputs
from the seeded generators in ``workloads``.

Attention and block mass are the plain definitions in ``kvs_oracle.c``.  The
scoring, tiering, selection, page assembly and demote/readmit bookkeeping are
written here with numpy, in fp64, each operation in the order stated in its
docstring.

Sources (page titles and sections):
  [VA]  "KV-Cache Offloading for LLM Inference -- Visual Reference" (v6.0):
        s.3 KV-cache size formula; s.11 EMA update rule, Diagram 11.2 worked
        example and half-life; s.12 priority P and tier thresholds.
  [GQA] "GQA per-head attention as scoring streams" figure page: 640
        streams aggregated into one score per (sequence, 16-token block);
        64-byte per-block record; identity key and score persist across
        eviction and are restored on re-admission.
  [ARCH] "LLM KV cache offload" architecture page: block manager, block
        tables, reference counts for shared blocks, pinned-host staging.
  [VA]  s.14 "Prefetching Strategy", Diagram 14.1: the prefetch targets
        (anchor zone, recent window, high EMA); s.12 notes beside the P
        formula: prefetch priority 1/(1 + distance/100) and the fetch-order
        blend 0.6 rope_factor + 0.4 ema_factor.
  [KIVI] "Fitting a Million Tokens" s.02 "Quantize the cache": E4M3 pages;
        2-bit keys per channel in 32-token groups, values per token, fp16
        scale and zero per group, an unquantised residual window.
  [RETR] "RETRACTIONS": s.3 brute-force argmin audit of victim selection;
        the lazily decayed EMA and its order-preserving key
        K = ln S_touch + t_touch*(-ln(1-alpha)).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_BUILD = _HERE / "_build"
_SO = _BUILD / "liboracle.so"
_lib = None

# ---------------------------------------------------------------------------
# build / load
# ---------------------------------------------------------------------------


def build(force: bool = False) -> Path:
    """Compile kvs_oracle.c into a shared library (gcc, IEEE fp64 order)."""
    src = _HERE / "kvs_oracle.c"
    _BUILD.mkdir(exist_ok=True)
    if force or not _SO.exists() or _SO.stat().st_mtime < src.stat().st_mtime:
        tmp = _SO.with_suffix(f".tmp{os.getpid()}.so")
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", str(src), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_SO))
        P = ctypes.c_void_p
        lib.orc_decode_heads.argtypes = [
            P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, P]
        lib.orc_decode_heads.restype = ctypes.c_int
        lib.orc_decode_heads_u8.argtypes = [
            P, P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, P]
        lib.orc_decode_heads_u8.restype = ctypes.c_int
        lib.orc_decode_heads_f32.argtypes = [
            P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, P]
        lib.orc_decode_heads_f32.restype = ctypes.c_int
        lib.orc_aggregate_mass.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, P]
        lib.orc_aggregate_mass.restype = None
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 bit array (numpy) -> contiguous uint16."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # plain CPU conversion of the bit pattern only
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# attention and block mass (C)
# ---------------------------------------------------------------------------


def decode(q, K, V, *, L, Hq, Hkv, d, block_tokens=16, heads=None,
           threads=None, want_out=True, want_head_mass=True, k_lut=None, v_lut=None):
    """Decode attention of one sequence.

    q: [L][Hq][d] bf16; K, V: [n][L][Hkv][d] bf16 in logical token order,
    float32 numpy arrays (values), or uint8 codes with k_lut / v_lut (256
    values each, e.g. e4m3_lut(scale)).
    heads: iterable of flat l*Hq+h indices (None = all, in order).
    Returns dict(out [nh][d], lse [nh], head_mass [nh][nb] or None).
    """
    lib = _load()
    coded = k_lut is not None
    f32 = isinstance(K, np.ndarray) and K.dtype == np.float32
    qb = _u16(q)
    if f32:
        kb = np.ascontiguousarray(K)
        vb = np.ascontiguousarray(np.asarray(V, np.float32))
    elif coded:
        kb = np.ascontiguousarray(np.asarray(K, np.uint8))
        vb = np.ascontiguousarray(np.asarray(V, np.uint8))
        lk = np.ascontiguousarray(np.asarray(k_lut, np.float64))
        lv = np.ascontiguousarray(np.asarray(v_lut, np.float64))
        assert lk.shape == (256,) and lv.shape == (256,)
    else:
        kb, vb = _u16(K), _u16(V)
    n = kb.shape[0]
    assert qb.shape == (L, Hq, d) and kb.shape == (n, L, Hkv, d) and vb.shape == kb.shape
    nb = (n + block_tokens - 1) // block_tokens
    hl = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    nh = L * Hq if hl is None else len(hl)
    out = np.zeros((nh, d), np.float64) if want_out else None
    lse = np.zeros(nh, np.float64)
    hm = np.zeros((nh, nb), np.float64) if want_head_mass else None
    hp = _ptr(hl) if hl is not None else None
    nt = int(threads or os.cpu_count() or 1)
    if f32:
        rc = lib.orc_decode_heads_f32(_ptr(qb), _ptr(kb), _ptr(vb), n, L, Hq, Hkv, d,
                                      block_tokens, hp, nh, nt, _ptr(out), _ptr(lse), _ptr(hm))
    elif coded:
        rc = lib.orc_decode_heads_u8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(lk), _ptr(lv), n, L, Hq,
                                     Hkv, d, block_tokens, hp, nh, nt, _ptr(out), _ptr(lse), _ptr(hm))
    else:
        rc = lib.orc_decode_heads(_ptr(qb), _ptr(kb), _ptr(vb), n, L, Hq, Hkv, d,
                                  block_tokens, hp, nh, nt, _ptr(out), _ptr(lse), _ptr(hm))
    if rc != 0:
        raise RuntimeError("oracle decode failed (bad argument or out of memory)")
    return {"out": out, "lse": lse, "head_mass": hm}


def aggregate_mass(head_mass: np.ndarray, *, L, Hq, Hkv) -> np.ndarray:
    """M(b) from all L*Hq per-head block masses [L*Hq][nb] ([GQA] s.2)."""
    lib = _load()
    hm = np.ascontiguousarray(head_mass, dtype=np.float64)
    assert hm.shape[0] == L * Hq
    nb = hm.shape[1]
    mass = np.zeros(nb, np.float64)
    lib.orc_aggregate_mass(_ptr(hm), nb, L, Hq, Hkv, _ptr(mass))
    return mass


def decode_with_mass(q, K, V, *, L, Hq, Hkv, d, block_tokens=16, threads=None,
                     want_out=True, k_lut=None, v_lut=None):
    """All heads of one sequence: out [L][Hq][d], lse [L][Hq], mass [nb]."""
    r = decode(q, K, V, L=L, Hq=Hq, Hkv=Hkv, d=d, block_tokens=block_tokens,
               threads=threads, want_out=want_out, want_head_mass=True, k_lut=k_lut, v_lut=v_lut)
    mass = aggregate_mass(r["head_mass"], L=L, Hq=Hq, Hkv=Hkv)
    return {
        "out": None if r["out"] is None else r["out"].reshape(L, Hq, d),
        "lse": r["lse"].reshape(L, Hq),
        "head_mass": r["head_mass"],
        "mass": mass,
    }


# ---------------------------------------------------------------------------
# FP8 E4M3 codes ("Fitting a Million Tokens", s.02: FP8 E4M3 KV halves the
# bytes).  Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no
# infinities; S.1111.111 is NaN; largest finite 448, smallest subnormal 2^-9.
# ---------------------------------------------------------------------------


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 codes (NaN for the two NaN codes)."""
    v = np.empty(256, np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 15 and m == 7:
            v[c] = np.nan
        elif e == 0:
            v[c] = sign * 2.0 ** -6 * (m / 8.0)
        else:
            v[c] = sign * 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return v


_E4M3 = e4m3_values()
_E4M3_POS = _E4M3[:127]          # codes 0..126: 0 .. 448, increasing


def e4m3_lut(scale: float) -> np.ndarray:
    """Dequantised value of each code: code value x scale (float64)."""
    return _E4M3 * np.float64(np.float32(scale))


def quantize_e4m3(x, scale: float) -> np.ndarray:
    """Codes of x / scale: the division in IEEE fp32, then the nearest code
    (ties to the even mantissa), magnitudes beyond 448 saturating to 448,
    the sign kept (also for results that round to zero)."""
    xf = np.asarray(x, np.float32)
    y = (xf / np.float32(scale)).astype(np.float64)
    a = np.minimum(np.abs(y), 448.0)
    hi = np.searchsorted(_E4M3_POS, a)                 # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)


def quantize_bf16_e4m3(bits, scale: float) -> np.ndarray:
    """quantize_e4m3 of bf16 bit patterns (a torch bf16 tensor or uint16)."""
    return quantize_e4m3(bf16_to_f64(_u16(bits)).astype(np.float32), scale)


# ---------------------------------------------------------------------------
# KIVI-style 2-bit groups ([KIVI] s.02 "Quantize the cache": keys per channel
# in groups of 32 tokens, two 16-token blocks; values per token in groups of
# 32 channels; asymmetric, an fp16 scale and zero per group; the newest ~128
# tokens stay unquantised, the boundary snapped down to a whole group)
# ---------------------------------------------------------------------------

KIVI_GROUP = 32
KIVI_RESIDUAL = 128
KIVI_TILE_BYTES = 3072      # one (layer, KV head) of a 32-token group, d = 128


def kivi_quantized_tokens(n: int, residual: int = KIVI_RESIDUAL, group: int = KIVI_GROUP) -> int:
    """Tokens in whole quantised groups: every group of 32 that ends at least
    `residual` tokens before the end, group * floor(max(0, n - residual) / group)."""
    return group * (max(0, n - residual) // group)


def kivi_quant(x):
    """Asymmetric 2-bit quantisation along the last axis (one group).

    x: float32 (bf16 values widened exactly).  In fp32, rounded as written:
    mn, mx = min, max; scale = fp16(fp32(mx - mn) / 3); zero = fp16(mn);
    code = clamp(rint(fp32(x - zero) / scale), 0, 3) (ties to even), 0 where
    scale is 0.  Returns (codes uint8, scale f16, zero f16)."""
    x = np.asarray(x, np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    scale = ((mx - mn) / np.float32(3.0)).astype(np.float16)
    zero = mn.astype(np.float16)
    sf = scale.astype(np.float32)[..., None]
    zf = zero.astype(np.float32)[..., None]
    t = x - zf
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(sf > 0, t / np.where(sf > 0, sf, np.float32(1.0)), np.float32(0.0))
    codes = np.clip(np.rint(u), 0, 3).astype(np.uint8)
    return codes, scale, zero


def kivi_dequant(codes, scale, zero) -> np.ndarray:
    """fp16(code * scale + zero), one rounding (the product and sum are exact
    in fp64).  scale and zero broadcast over the group axis (last)."""
    v = (np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[..., None]
         + np.asarray(zero, np.float64)[..., None])
    return v.astype(np.float16)


def kivi_quant_k(Kg):
    """Keys of one group, [32][L][Hkv][d] (bf16 bits or float32): per
    channel over the 32 tokens.  Returns codes [32][L][Hkv][d], scale and
    zero [L][Hkv][d]."""
    x = _as_f32(Kg)
    c, s, z = kivi_quant(np.moveaxis(x, 0, -1))
    return np.moveaxis(c, -1, 0), s, z


def kivi_quant_v(Vg):
    """Values of one group, [32][L][Hkv][d]: per token over groups of 32
    channels.  Returns codes [32][L][Hkv][d], scale and zero
    [32][L][Hkv][d/32]."""
    x = _as_f32(Vg)
    n, L, H, d = x.shape
    c, s, z = kivi_quant(x.reshape(n, L, H, d // KIVI_GROUP, KIVI_GROUP))
    return c.reshape(n, L, H, d), s, z


def _as_f32(x) -> np.ndarray:
    if isinstance(x, np.ndarray) and x.dtype == np.float32:
        return x
    return bf16_to_f64(_u16(x)).astype(np.float32)


def kivi_effective(K, V):
    """K, V of one sequence ([n][L][Hkv][d] bf16) as attention sees them
    under the 2-bit scheme: tokens before kivi_quantized_tokens(n)
    dequantised from their groups, the rest as stored.  float32 arrays."""
    Kf, Vf = _as_f32(K).copy(), _as_f32(V).copy()
    n = Kf.shape[0]
    for a in range(0, kivi_quantized_tokens(n), KIVI_GROUP):
        b = a + KIVI_GROUP
        ck, sk, zk = kivi_quant_k(Kf[a:b])
        Kf[a:b] = np.moveaxis(kivi_dequant(np.moveaxis(ck, 0, -1), sk, zk), -1, 0).astype(np.float32)
        cv, sv, zv = kivi_quant_v(Vf[a:b])
        n_, L, H, d = cv.shape
        Vf[a:b] = kivi_dequant(cv.reshape(n_, L, H, d // KIVI_GROUP, KIVI_GROUP), sv, zv) \
            .reshape(n_, L, H, d).astype(np.float32)
    return Kf, Vf


def kivi_group_tile(ck, sk, zk, cv, sv, zv) -> bytes:
    """Bytes of one (layer, KV head) of a group page (d = 128), the layout a
    warp of the decode kernel reads (lane = 4*g + t, g = lane // 4, t = lane % 4).

    Code words hold operand pairs as the two 2-bit fields of a byte's two
    nibbles: in byte k (k = 0..3) of word w, the pair (bits 0-1, bits 4-5)
    belongs to operand register k of step 2w and the pair (bits 2-3,
    bits 6-7) to register k of step 2w + 1 (first element in the low field).

      K codes  [0, 1024)   : [block j][lane][word w in 0..3]; step s = k-step
                             (16 channels) s, register r: token 16j + g +
                             8*(r % 2), channels (c, c + 8) for r < 2 and
                             (c + 1, c + 9) for r >= 2, c = 32t + 16*(s // 4)
                             + 2*(s % 4).
      V codes  [1024, 2048): [block j][lane][word w]; step s = m-tile
                             (16 channels) s, register r: channel 16s + g +
                             8*(r % 2), tokens (16j + 2t + 8*(r // 2), the next).
      K meta   [2048, 2560): [half h in 0..1][ip in 0..3][t] of (scale pair,
                             zero pair) for i = 2ip, then for i = 2ip + 1;
                             each pair two fp16: channel 32t + 16h + i
                             (low), that channel + 8 (high).
      V meta   [2560, 2816): scale pairs [block j][token pair p in 0..7]
                             [channel group c in 0..3]: tokens 16j + 2p
                             (low) and 16j + 2p + 1 (high);
               [2816, 3072): zero pairs, the same order.
      Every scale is stored doubled, 2 * scale (exact in fp16).

    ck, cv: codes [32][d]; sk, zk: [d]; sv, zv: [32][d/32]."""
    ck = np.asarray(ck, np.uint32)
    cv = np.asarray(cv, np.uint32)

    def k_pair(j, g, t, s, r):
        tok = 16 * j + g + 8 * (r % 2)
        c = 32 * t + 16 * (s // 4) + 2 * (s % 4) + (r // 2)
        return ck[tok, c], ck[tok, c + 8]

    def v_pair(j, g, t, s, r):
        ch = 16 * s + g + 8 * (r % 2)
        tok = 16 * j + 2 * t + 8 * (r // 2)
        return cv[tok, ch], cv[tok + 1, ch]

    def words(pair):
        out = np.zeros((2, 32, 4), np.uint32)
        for j in range(2):
            for lane in range(32):
                g, t = lane // 4, lane % 4
                for w in range(4):
                    word = 0
                    for k in range(4):
                        for half, s in ((0, 2 * w), (1, 2 * w + 1)):
                            lo, hi = pair(j, g, t, s, k)
                            word |= int(lo) << (8 * k + 2 * half)
                            word |= int(hi) << (8 * k + 4 + 2 * half)
                    out[j, lane, w] = word
        return out

    kc, vc = words(k_pair), words(v_pair)
    f16 = lambda a: np.asarray(a, np.float16).view(np.uint16).astype(np.uint32)
    two = np.float16(2.0)
    skb, zkb = f16(np.asarray(sk, np.float16) * two), f16(zk)
    km = np.zeros((2, 4, 4, 2, 2), np.uint32)
    for h in range(2):
        for ip in range(4):
            for t in range(4):
                for di in range(2):
                    ch = 32 * t + 16 * h + 2 * ip + di
                    km[h, ip, t, di, 0] = skb[ch] | (skb[ch + 8] << 16)
                    km[h, ip, t, di, 1] = zkb[ch] | (zkb[ch + 8] << 16)
    svb, zvb = f16(np.asarray(sv, np.float16) * two), f16(zv)
    vm = np.zeros((2, 2, 8, 4), np.uint32)        # [scales, zeros][j][p][c]
    for j in range(2):
        for p_ in range(8):
            for c in range(4):
                a = 16 * j + 2 * p_
                vm[0, j, p_, c] = svb[a, c] | (svb[a + 1, c] << 16)
                vm[1, j, p_, c] = zvb[a, c] | (zvb[a + 1, c] << 16)
    out = b"".join(x.astype("<u4").tobytes() for x in (kc, vc, km, vm))
    assert len(out) == KIVI_TILE_BYTES
    return out


def kivi_group_page(Kg, Vg) -> bytes:
    """Bytes of one group page: the tiles of all (layer, KV head), layer
    outermost, for the 32 tokens Kg, Vg ([32][L][Hkv][128])."""
    ck, sk, zk = kivi_quant_k(Kg)
    cv, sv, zv = kivi_quant_v(Vg)
    L, H = ck.shape[1], ck.shape[2]
    return b"".join(kivi_group_tile(ck[:, l, h], sk[l, h], zk[l, h], cv[:, l, h], sv[:, l, h], zv[:, l, h])
                    for l in range(L) for h in range(H))


# ---------------------------------------------------------------------------
# 64-byte per-block record ([GQA]: 16 B identity key, 8 B score, 8 B touch
# timestamp, 4 B touch count, reserved).  The reserved bytes carry the tier,
# the last priority, the last mass and the event-driven (LRFU) score at the
# last touch, so that every step can be compared.
# ---------------------------------------------------------------------------

REC_DTYPE = np.dtype({
    "names": ["seq_id", "block_idx", "score", "last_touch", "count", "tier",
              "flags", "pad0", "prio", "mass", "rsv", "lrfu"],
    "formats": ["<u8", "<u8", "<f8", "<u8", "<u4", "u1", "u1", "<u2", "<f8",
                "<f4", ("u1", 4), "<f8"],
    "offsets": [0, 8, 16, 24, 32, 36, 37, 38, 40, 48, 52, 56],
    "itemsize": 64,
})
TIER_UNSCORED = 255


def new_records(seq_id: int, first_block: int, count: int, t_create: int) -> np.ndarray:
    """Records of freshly opened blocks: score 0 (the worked example of [VA]
    Diagram 11.2 starts from 0), last touch = creation step, count 0."""
    r = np.zeros(count, REC_DTYPE)
    r["seq_id"] = seq_id
    r["block_idx"] = np.arange(first_block, first_block + count, dtype=np.uint64)
    r["last_touch"] = t_create
    r["tier"] = TIER_UNSCORED
    return r


def ema(prev: np.ndarray, attn: np.ndarray, alpha: float) -> np.ndarray:
    """[VA] s.11: score_t = alpha*attention_t + (1-alpha)*score_{t-1}.
    Evaluated as (alpha*attn) + ((1.0-alpha)*prev) in fp64."""
    a = np.float64(alpha)
    return a * np.asarray(attn, np.float64) + (np.float64(1.0) - a) * np.asarray(prev, np.float64)


def lrfu_decay(alpha: float, dt) -> np.ndarray:
    """(1 - alpha)^dt for integer dt >= 0 by binary exponentiation in fp64:
    result = 1, base = 1 - alpha; for each bit of dt from the lowest: if set,
    result = result * base; then base = base * base."""
    dt = np.asarray(dt, np.int64).copy()
    base = np.full(dt.shape, np.float64(1.0) - np.float64(alpha))
    res = np.ones(dt.shape, np.float64)
    while np.any(dt > 0):
        odd = (dt & 1) == 1
        res = np.where(odd, res * base, res)
        base = base * base
        dt >>= 1
    return res


def lrfu_touch(S_prev, t_prev, t: int, alpha: float) -> np.ndarray:
    """Event-driven score of a block touched at step t ([RETR] s.3 lazy
    decay; the [VA] s.11 EMA of the touch indicator x: score_t = alpha*x_t +
    (1-alpha)*score_{t-1}, with x = 0 between touches).  S_prev is the score
    right after the previous touch at t_prev (0 and the creation step for a
    block never touched): S = alpha + (1-alpha)^(t - t_prev) * S_prev, the
    product first."""
    d = lrfu_decay(alpha, np.int64(t) - np.asarray(t_prev, np.int64))
    return np.float64(alpha) + d * np.asarray(S_prev, np.float64)


def lrfu_decayed(S_touch, t_touch, t: int, alpha: float) -> np.ndarray:
    """The score at step t of a block last touched at t_touch: S_touch *
    (1-alpha)^(t - t_touch)."""
    return np.asarray(S_touch, np.float64) * lrfu_decay(alpha, np.int64(t) - np.asarray(t_touch, np.int64))


# the double nearest ln 2, and the double nearest sqrt(1/2)
LN2 = float.fromhex("0x1.62e42fefa39efp-1")
SQRT_HALF = float.fromhex("0x1.6a09e667f3bcdp-1")
LN_SERIES_TERMS = 12      # odd powers s^1 .. s^23


def ln_series(x) -> np.ndarray:
    """Natural logarithm of positive normal fp64 values from its series
    definition: x = m * 2^e with m in [sqrt(1/2), sqrt(2)) (m from frexp,
    doubled below sqrt(1/2)); s = (m - 1)/(m + 1), z = s*s;
    ln m = 2 artanh(s) = 2 s (1 + z/3 + z^2/5 + ... + z^11/23), the
    bracket by Horner's rule from the 1/23 term down (h = 1/d + z*h);
    ln x = e*ln2 + ln m.  |s| < 0.172, so the series is cut where its next
    term is below 1e-20 of the first.  Every step is one IEEE fp64 operation
    (no fused multiply-add), so any program taking the same steps gets the
    same bits: the logarithm in the LRFU key must order near-equal keys the
    same way wherever it is evaluated.  (The series: Abramowitz and Stegun,
    Handbook of Mathematical Functions, 4.1.27.)"""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    low = m < SQRT_HALF
    m = np.where(low, m * 2.0, m)
    e = np.where(low, e - 1, e).astype(np.float64)
    s = (m - 1.0) / (m + 1.0)
    z = s * s
    h = np.full(x.shape, 1.0 / (2 * LN_SERIES_TERMS - 1))
    for d in range(2 * LN_SERIES_TERMS - 3, 0, -2):
        h = (1.0 / d) + z * h
    return e * LN2 + 2.0 * (s * h)


def lrfu_slope(alpha: float) -> float:
    """-ln(1 - alpha), by ln_series: the key's growth per step of t_touch."""
    return float(-ln_series(np.float64(1.0) - np.float64(alpha)))


def lrfu_key(S_touch, t_touch, alpha: float) -> np.ndarray:
    """[RETR] s.3 order-preserving key K = ln S_touch + t_touch*(-ln(1-alpha)):
    ln of the decayed score at any t is K + t*ln(1-alpha), so K orders the
    blocks as the decayed score does, at every t (-inf for S_touch = 0).
    Both logarithms by ln_series; the sum and product in fp64 as written."""
    S = np.asarray(S_touch, np.float64)
    pos = S > 0
    lnS = np.where(pos, ln_series(np.where(pos, S, 1.0)), -np.inf)
    return lnS + np.asarray(t_touch, np.float64) * lrfu_slope(alpha)


def recency(t: int, last_touch: np.ndarray, W: int) -> np.ndarray:
    """R = 1 - (t - last_touch)/W, clipped to [0, 1]: 1.0 - (age / W)."""
    age = (np.int64(t) - np.asarray(last_touch, np.int64)).astype(np.float64)
    r = np.float64(1.0) - age / np.float64(W)
    return np.minimum(np.maximum(r, 0.0), 1.0)


def priority(R, E, N, weights=(0.25, 0.55, 0.20)) -> np.ndarray:
    """[VA] s.12: P = 0.25*R + 0.55*E + 0.20*N, summed left to right."""
    wR, wE, wN = (np.float64(w) for w in weights)
    return (wR * np.asarray(R, np.float64) + wE * np.asarray(E, np.float64)) + wN * np.asarray(N, np.float64)


def tier_of(P, cuts=(0.3, 0.6)) -> np.ndarray:
    """[VA] Diagram 12.2, boundaries half-open: P < 0.3 -> 2 (lowest tier),
    0.3 <= P < 0.6 -> 1, P >= 0.6 -> 0 (pinned)."""
    lo, hi = np.float64(cuts[0]), np.float64(cuts[1])
    P = np.asarray(P, np.float64)
    return np.where(P >= hi, 0, np.where(P >= lo, 1, 2)).astype(np.uint8)


def score_update(rec: np.ndarray, mass: np.ndarray, t: int, alpha: float,
                 W: int = 64, weights=(0.25, 0.55, 0.20), cuts=(0.3, 0.6)) -> np.ndarray:
    """One scoring step over the nb records (block order) of one sequence.

    mass: the step's M(b), float64 (or float32, widened exactly).
    Order: EMA -> touch (mass >= 1/num_blocks: M*nb >= 1, count += 1,
    the event-driven score by lrfu_touch, last_touch = t) -> recency R ->
    anchor N (block 0 and the newest block) -> P -> tier.  Returns a new
    record array.
    """
    r = rec.copy()
    nb = len(r)
    M = np.asarray(mass, dtype=np.float64)
    assert M.shape == (nb,)
    r["score"] = ema(r["score"], M, alpha)
    touched = M * np.float64(nb) >= 1.0
    r["count"] = r["count"] + touched.astype(np.uint32)
    r["lrfu"] = np.where(touched, lrfu_touch(r["lrfu"], r["last_touch"], t, alpha), r["lrfu"])
    r["last_touch"] = np.where(touched, np.uint64(t), r["last_touch"])
    R = recency(t, r["last_touch"], W)
    N = np.zeros(nb, np.float64)
    if nb:
        N[0] = 1.0
        N[nb - 1] = 1.0
    P = priority(R, r["score"], N, weights)
    r["prio"] = P
    r["tier"] = tier_of(P, cuts)
    r["mass"] = M.astype(np.float32)
    return r


# ---------------------------------------------------------------------------
# selection ([VA] s.12 tiers; [RETR] s.3 brute-force audit)
# ---------------------------------------------------------------------------


def _ordered(recs_by_seq: dict) -> np.ndarray:
    """All records in ascending (seq_id, block_idx) order."""
    parts = [recs_by_seq[s] for s in sorted(recs_by_seq)]
    return np.concatenate(parts) if parts else np.zeros(0, REC_DTYPE)


def select_thresh(recs_by_seq: dict) -> list:
    """Every record in the lowest tier (P < 0.3), ascending (seq_id, block_idx)."""
    allr = _ordered(recs_by_seq)
    pick = allr["tier"] == 2
    return [(int(a), int(b)) for a, b in zip(allr["seq_id"][pick], allr["block_idx"][pick])]


def lowfrac_k(n_records: int, frac: float) -> int:
    return int(math.floor(np.float64(frac) * np.float64(n_records)))


def select_lowfrac(recs_by_seq: dict, frac: float) -> list:
    """The k = floor(frac*N) records of smallest P, ties broken by
    (seq_id, block_idx); returned in ascending (seq_id, block_idx) order.
    Plain full sort of every record."""
    allr = _ordered(recs_by_seq)
    k = lowfrac_k(len(allr), frac)
    order = sorted(range(len(allr)), key=lambda i: (float(allr["prio"][i]), i))
    chosen = sorted(order[:k])
    return [(int(allr["seq_id"][i]), int(allr["block_idx"][i])) for i in chosen]


def select_lrfu(recs_by_seq: dict, frac: float, alpha: float) -> list:
    """The k = floor(frac*N) records of smallest LRFU key (lrfu_key of the
    score at the last touch and last_touch), ties broken by (seq_id,
    block_idx); returned in ascending (seq_id, block_idx) order."""
    allr = _ordered(recs_by_seq)
    k = lowfrac_k(len(allr), frac)
    K = lrfu_key(allr["lrfu"], allr["last_touch"], alpha)
    order = sorted(range(len(allr)), key=lambda i: (float(K[i]), i))
    chosen = sorted(order[:k])
    return [(int(allr["seq_id"][i]), int(allr["block_idx"][i])) for i in chosen]


def lrfu_victims_brute_force(recs_by_seq: dict, frac: float, t: int, alpha: float) -> list:
    """[RETR] s.3 audit: the k = floor(frac*N) records of smallest decayed
    score at step t, each computed directly (lrfu_decayed), ties broken by
    (seq_id, block_idx); ascending (seq_id, block_idx)."""
    allr = _ordered(recs_by_seq)
    k = lowfrac_k(len(allr), frac)
    S = lrfu_decayed(allr["lrfu"], allr["last_touch"], t, alpha)
    order = sorted(range(len(allr)), key=lambda i: (float(S[i]), i))
    chosen = sorted(order[:k])
    return [(int(allr["seq_id"][i]), int(allr["block_idx"][i])) for i in chosen]


# ---------------------------------------------------------------------------
# page assembly and gather ([ARCH]: one block = one page of all layers and
# KV heads, laid out contiguously for coalesced transfer)
# ---------------------------------------------------------------------------


def assemble_page(K_blk, V_blk, block_tokens: int = 16) -> bytes:
    """Bytes of one page from the logical K, V of its t <= block_tokens
    tokens ([t][L][Hkv][d] each: bf16, or uint8 codes for FP8 pages).

    Layout, outermost first: layer, {K, V}, KV head, token slot, head dim;
    bf16 little-endian or one byte per code; slots past the last token are
    zero.
    """
    if isinstance(K_blk, np.ndarray) and K_blk.dtype == np.uint8:
        kb, vb = K_blk, V_blk
        t, L, Hkv, d = kb.shape
        page = np.zeros((L, 2, Hkv, block_tokens, d), np.uint8)
        page[:, 0, :, :t, :] = kb.transpose(1, 2, 0, 3)
        page[:, 1, :, :t, :] = vb.transpose(1, 2, 0, 3)
        return page.tobytes()
    kb, vb = _u16(K_blk), _u16(V_blk)
    t, L, Hkv, d = kb.shape
    assert t <= block_tokens and vb.shape == kb.shape
    page = np.zeros((L, 2, Hkv, block_tokens, d), np.uint16)
    page[:, 0, :, :t, :] = kb.transpose(1, 2, 0, 3)
    page[:, 1, :, :t, :] = vb.transpose(1, 2, 0, 3)
    return page.tobytes()


def gather_plan(selected: list, page_of: dict, refs_of: dict) -> list:
    """Pages to gather for a selected list of (seq_id, block_idx) keys.

    page_of[key] -> page identity; refs_of[page] -> set of keys referencing
    it.  A page is gathered when every record referencing it is selected
    (a shared block is released only by its last user, [ARCH] reference
    counts), once, at the position of its first selected record.
    Returns the page identities in gather order.
    """
    sel = set(selected)
    seen, plan = set(), []
    for key in selected:
        p = page_of[key]
        if p in seen:
            continue
        if refs_of[p] <= sel:
            plan.append(p)
            seen.add(p)
    return plan


# ---------------------------------------------------------------------------
# identity-keyed demote / readmit ([GQA]: identity key and score persist and
# are restored on re-admission rather than reset)
# ---------------------------------------------------------------------------


class IdentityStore:
    """Key (seq_id, block_idx) -> (64-byte record, page bytes)."""

    def __init__(self):
        self._m = {}

    def demote(self, key, record: np.ndarray, page: bytes):
        if key in self._m:
            raise KeyError(f"{key} already demoted")
        self._m[key] = (record.copy(), bytes(page))

    def readmit(self, key):
        if key not in self._m:
            raise KeyError(f"{key} not demoted")
        return self._m.pop(key)

    def __contains__(self, key):
        return key in self._m

    def __len__(self):
        return len(self._m)


# ---------------------------------------------------------------------------
# prefetch order of demoted blocks ([VA] s.14 Diagram 14.1; s.12 notes)
# ---------------------------------------------------------------------------

ANCHOR_LAST_POSITION = 100    # anchor zone: token positions 0..100
RECENT_WINDOW = 200           # recent window: positions m-200..m-1


def prefetch_class(block_idx: int, ntok: int, block_tokens: int = 16) -> int:
    """0 if the block holds a position of the anchor zone [0, 100], else 1 if
    it holds a position of the recent window [m - 200, m - 1] (m = the
    sequence's token count), else 2: the order of the three target lists."""
    first = block_idx * block_tokens
    last = first + block_tokens - 1
    if first <= ANCHOR_LAST_POSITION:
        return 0
    if last >= ntok - RECENT_WINDOW:
        return 1
    return 2


def rope_factor(distance: int) -> float:
    """1 / (1 + distance / 100), in fp64: division, addition, division."""
    return 1.0 / (1.0 + float(distance) / 100.0)


def prefetch_blend(block_idx: int, ntok: int, ema_score: float, block_tokens: int = 16) -> float:
    """0.6 rope_factor + 0.4 ema_factor.  distance = tokens between the last
    token (position m - 1) and the block's last position (0 when the block
    holds the last token); ema_factor = the block's EMA score E as kept in
    its record.  fp64: two products, then their sum."""
    last = block_idx * block_tokens + block_tokens - 1
    distance = max(0, (ntok - 1) - last)
    return 0.6 * rope_factor(distance) + 0.4 * float(ema_score)


def prefetch_order(cands, budget: int, block_tokens: int = 16) -> list:
    """Fetch order of demoted blocks: class ascending, blend descending, then
    (seq_id, block_idx) ascending; the first `budget` entries.

    cands: iterable of (seq_id, block_idx, ntok, ema_score).
    Returns [(seq_id, block_idx, class, blend)]."""
    rows = []
    for seq_id, b, m, e in cands:
        blend = min(prefetch_blend(b, m, e, block_tokens), 1.0)
        rows.append((prefetch_class(b, m, block_tokens), -blend, int(seq_id), int(b)))
    rows.sort()
    return [(sid, b, c, -nb) for c, nb, sid, b in rows[:budget]]


# ---------------------------------------------------------------------------
# capacity arithmetic ([VA] s.3; [GQA] 64 B x blocks)
# ---------------------------------------------------------------------------


def kv_bytes_per_token(L, Hkv, d, elem_bytes=2) -> int:
    """2 (K and V) x layers x KV heads x head dim x bytes per element."""
    return 2 * L * Hkv * d * elem_bytes


def metadata_bytes(num_blocks: int, record_bytes: int = 64) -> int:
    return num_blocks * record_bytes
