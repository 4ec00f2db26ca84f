"""CPU oracle for the CSA2 compressed-sparse-attention hot path.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the bench's
CPU-baseline / reference leg may import or run this module.  The CUDA library
never calls it, and it shares no code, header, table or constant generator with
the CUDA sources.

Plain numpy in float64 (bf16, fp32 and dequantised FP4 inputs are exact in f64).
Where a step has a plain definition it is written out directly; a library
primitive (matmul, sort, exp) may serve as one step.  No blocking, fusion or
reordering beyond what the definitions state.

Sources (three web pages on CSA / CSA2), cited below by short title:
  * «CSA2：跨层共享的压缩稀疏注意力» (daiw.org)                 -> "CSA2 page"
  * «DeepSeek 的 Attention 演进 -【DSA、CSA、CSA2】» (0xnullpath) -> "Attention-evolution page"
  * «从 DSA 到 CSA/HCA：先压缩时间轴，再决定怎样寻址» (wineandchord) -> "DSA-to-CSA/HCA page"

Readings taken where the pages are silent (each repeated at its function):
  * indexer score has no scale and no softmax (eq. 16 has none);
  * causal rule t >= m(j+1), i.e. floor(t/m) entries are visible;
  * top-k ties: lower entry index wins; fewer than k visible: all are returned;
  * pool: newest visible block always kept, the other slots by (block max desc,
    block asc); a partial last block scores over its visible members only;
  * RMSNorm: x / sqrt(mean(x^2) + 1e-6), unit gain, over all 512 channels;
  * RoPE: last 64 dims as interleaved pairs (448+2j, 449+2j), theta_j =
    10000^(-2j/64), angle in f64; compressed entry i sits at position pos0 + m*i;
    stored rows are already rotated at their own position;
  * FP4 main KV: 16-channel E4M3 scale s = E4M3_RNE(f32(amax)/6), codes
    E2M1_RNE(f32(x)/s) (IEEE f32 divisions), channel 2i in the low nibble, 256
    code bytes then 32 scale bytes; s == 0 -> all codes 0;
  * MXFP4 indexer K: OCP MX rule, scale 2^(floor(log2 amax) - 2) as E8M0, 64
    code bytes then 4 scale bytes; amax == 0 -> scale byte 0, codes 0;
  * E2M1 rounding is round-to-nearest-even with saturation at +-6, sign kept.

Pins (tests that tie this code to something other than itself): the pages'
worked compressor example (y0 = 1, y1 = 2.5) and sparse shared-KV example; the
890 bytes-per-token table; m = 1 identity; equal logits -> mean; the two overlap
formulations agreeing; chunked == whole compression; exhaustive FP4 code tables
and the RNE tie table; E4M3 rounding against torch's float8_e4m3fn; brute-force
top-k / pool / dense-masked attention on tiny inputs; the pool-containment lemma;
sink = -inf -> mass 1; RMSNorm scale invariance; RoPE shift invariance.
The RoPE convention itself (pair layout, base, entry position) and the RMSNorm
epsilon are readings: parity unpinned for those constants (the invariants above
hold for any choice).
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

NEG_INF = -np.inf

# flag bits (same meaning as the library's, defined here independently)
QNORM, KVNORM, ROPE = 1, 2, 4
NORM_W, ROPE_W, PACK_W = 1, 2, 4
RMS_EPS = 1e-6
ROPE_DIMS = 64
ROPE_BASE = 10000.0


# =============================================================================
# Minifloat formats (OCP E2M1, E4M3 "FN", E8M0)
# Used by the FP4 main-KV format and the MXFP4 indexer-K format of the CSA2 page,
# section «890 字节是怎么来的».
# =============================================================================

def minifloat_decode(code, ebits: int, mbits: int, bias: int) -> np.ndarray:
    """Decode sign/exponent/mantissa bit fields to f64 (no inf/NaN handling)."""
    code = np.asarray(code, dtype=np.int64)
    m = code & ((1 << mbits) - 1)
    e = (code >> mbits) & ((1 << ebits) - 1)
    s = (code >> (mbits + ebits)) & 1
    frac = m.astype(np.float64) / (1 << mbits)
    normal = np.ldexp(1.0 + frac, (e - bias).astype(np.int64))
    subnormal = np.ldexp(frac, 1 - bias)
    mag = np.where(e > 0, normal, subnormal)
    return np.where(s == 1, -mag, mag)


def e2m1_decode(code) -> np.ndarray:
    """E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; 16 codes, max 6."""
    return minifloat_decode(code, 2, 1, 1)


def e4m3_decode(code) -> np.ndarray:
    """E4M3 (FN variant): bias 7, max 448, code 0x7F / 0xFF is NaN."""
    code = np.asarray(code, dtype=np.int64)
    v = minifloat_decode(code, 4, 3, 7)
    return np.where((code & 0x7F) == 0x7F, np.nan, v)


def e8m0_decode(code) -> np.ndarray:
    """E8M0 scale byte: 2^(code - 127); 0xFF is NaN."""
    code = np.asarray(code, dtype=np.int64)
    v = np.ldexp(1.0, code - 127)
    return np.where(code == 0xFF, np.nan, v)


def _rne_to_grid(x: np.ndarray, grid: np.ndarray, grid_codes: np.ndarray) -> np.ndarray:
    """Round |x| to the nearest value of an ascending non-negative grid; ties go to
    the code whose lowest bit (the mantissa lsb) is 0.  Values above the grid's top
    saturate to it.  Returns the magnitude codes."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.minimum(a, grid[-1])
    hi = np.searchsorted(grid, a, side="left")           # grid[hi] >= a
    hi = np.minimum(hi, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    even_hi = (grid_codes[hi] & 1) == 0
    pick_hi = np.where(tie, even_hi, pick_hi)
    return np.where(pick_hi, grid_codes[hi], grid_codes[lo])


_E2M1_CODES = np.arange(8, dtype=np.int64)
_E2M1_GRID = e2m1_decode(_E2M1_CODES)                   # 0, .5, 1, 1.5, 2, 3, 4, 6
_E4M3_CODES = np.arange(0x7F, dtype=np.int64)           # all finite non-negative codes
_E4M3_GRID = e4m3_decode(_E4M3_CODES)                   # 0 .. 448


def e2m1_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto E2M1, saturating at +-6, sign bit kept."""
    x = np.asarray(x, dtype=np.float64)
    mag = _rne_to_grid(x, _E2M1_GRID, _E2M1_CODES)
    sign = np.signbit(x).astype(np.int64)
    return (mag | (sign << 3)).astype(np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto E4M3 with saturation at +-448 (satfinite)."""
    x = np.asarray(x, dtype=np.float64)
    mag = _rne_to_grid(x, _E4M3_GRID, _E4M3_CODES)
    sign = np.signbit(x).astype(np.int64)
    return (mag | (sign << 7)).astype(np.uint8)


def nvfp4_row_bytes(c: int = 512) -> int:
    """Main-KV entry: c E2M1 codes (4 bits) + one E4M3 byte per 16 channels."""
    return c // 2 + c // 16


def mxfp4_row_bytes(d: int = 128) -> int:
    """Indexer-K entry: d E2M1 codes (4 bits) + one E8M0 byte per 32 values."""
    return d // 2 + d // 32


def _pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[rows, c] nibbles -> [rows, c/2] bytes, channel 2i in the low nibble."""
    codes = codes.astype(np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _unpack_nibbles(b: np.ndarray) -> np.ndarray:
    rows, half = b.shape
    out = np.empty((rows, 2 * half), dtype=np.uint8)
    out[:, 0::2] = b & 0x0F
    out[:, 1::2] = b >> 4
    return out


def nvfp4_pack(x) -> np.ndarray:
    """FP4 main-KV rows: per 16 channels s = E4M3_RNE(f32(amax)/6); if s == 0 all
    codes are 0, else code = E2M1_RNE(f32(x) / s) with IEEE f32 divisions.
    x: [rows, c] (values exact in f32) -> [rows, c/2 + c/16] uint8."""
    x = np.asarray(x, dtype=np.float32)
    rows, c = x.shape
    g = x.reshape(rows, c // 16, 16)
    amax = np.max(np.abs(g), axis=2).astype(np.float32)
    s_f32 = (amax / np.float32(6.0)).astype(np.float32)             # f32 RN division
    s_code = e4m3_encode(s_f32)
    s_val = e4m3_decode(s_code).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (g / s_val[:, :, None]).astype(np.float32)          # f32 RN division
    codes = e2m1_encode(ratio)
    codes = np.where((s_val == 0)[:, :, None], np.uint8(0), codes)
    return np.concatenate([_pack_nibbles(codes.reshape(rows, c)), s_code], axis=1)


def nvfp4_unpack(b, c: int = 512) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    codes = _unpack_nibbles(b[:, : c // 2])
    scales = e4m3_decode(b[:, c // 2: c // 2 + c // 16])
    vals = e2m1_decode(codes).reshape(b.shape[0], c // 16, 16) * scales[:, :, None]
    return vals.reshape(b.shape[0], c)


def mxfp4_pack(x) -> np.ndarray:
    """MXFP4 rows (OCP MX): per 32 values X = 2^(floor(log2 amax) - 2) stored as
    E8M0 (clamped to [0, 254]); code = E2M1_RNE(f32(x) / X); amax == 0 gives scale
    byte 0 and all codes 0.  x: [rows, d] -> [rows, d/2 + d/32] uint8."""
    x = np.asarray(x, dtype=np.float32)
    rows, d = x.shape
    g = x.reshape(rows, d // 32, 32)
    amax = np.max(np.abs(g), axis=2).astype(np.float64)
    _, ex = np.frexp(amax)                                # amax = f * 2^ex, f in [.5, 1)
    floor_log2 = ex.astype(np.int64) - 1
    code = np.clip(floor_log2 - 2 + 127, 0, 254)
    code = np.where(amax == 0, 0, code).astype(np.uint8)
    X = e8m0_decode(code).astype(np.float32)
    ratio = (g / X[:, :, None]).astype(np.float32)        # power of two: exact
    codes = e2m1_encode(ratio)
    codes = np.where((amax == 0)[:, :, None], np.uint8(0), codes)
    return np.concatenate([_pack_nibbles(codes.reshape(rows, d)), code], axis=1)


def mxfp4_unpack(b, d: int = 128) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    codes = _unpack_nibbles(b[:, : d // 2])
    scales = e8m0_decode(b[:, d // 2: d // 2 + d // 32])
    vals = e2m1_decode(codes).reshape(b.shape[0], d // 32, 32) * scales[:, :, None]
    return vals.reshape(b.shape[0], d)


# =============================================================================
# Gated token compressor
# =============================================================================

def _softmax_over_positions(logits: np.ndarray) -> np.ndarray:
    """Softmax along axis 0 (the candidate-position axis), separately per channel;
    rows at -inf get weight 0."""
    mx = np.max(logits, axis=0, keepdims=True)
    e = np.exp(logits - mx)
    return e / np.sum(e, axis=0, keepdims=True)


def compress(Ca, Za, m: int, Ba=None, Cb=None, Zb=None, Bb=None,
             prev_Cb=None, prev_Zb=None) -> np.ndarray:
    """Compressed entries E[i] of a token stream.

    Non-overlapping form (Attention-evolution page §4.1; DSA-to-CSA/HCA page eqs.
    22-23): per channel, a softmax over the m positions of block i of
    Z^a + B^a, and E[i] = sum_j S_j * C^a_j.

    Overlapping form (DSA-to-CSA/HCA page eqs. 11-12), used when Cb/Zb are given:
    the softmax runs per channel over 2m rows [Z^a_cur + B^a ; Z^b_prev + B^b] and
    E[i] = sum S^a (.) C^a_cur + sum S^b (.) C^b_prev.  The first block has no
    history: Z^b = -inf, C^b = 0, unless the previous block's (C^b, Z^b) is
    carried in (prev_Cb, prev_Zb), as the compressor's state cache does
    (Attention-evolution page §3.3).

    Shapes: Ca, Za, Cb, Zb [n, c]; Ba, Bb [m, c] (None -> 0); prev_* [m, c]."""
    Ca = np.asarray(Ca, dtype=np.float64)
    Za = np.asarray(Za, dtype=np.float64)
    n, c = Ca.shape
    if n % m:
        raise ValueError("n must be a multiple of m")
    Ba = np.zeros((m, c)) if Ba is None else np.asarray(Ba, dtype=np.float64)
    overlap = Cb is not None
    if overlap:
        Cb = np.asarray(Cb, dtype=np.float64)
        Zb = np.asarray(Zb, dtype=np.float64)
        Bb = np.zeros((m, c)) if Bb is None else np.asarray(Bb, dtype=np.float64)
        pC = np.zeros((m, c)) if prev_Cb is None else np.asarray(prev_Cb, dtype=np.float64)
        pZ = np.full((m, c), NEG_INF) if prev_Zb is None else np.asarray(prev_Zb, dtype=np.float64)
    out = np.empty((n // m, c))
    for i in range(n // m):
        cur = slice(m * i, m * (i + 1))
        if overlap:
            logits = np.concatenate([Za[cur] + Ba, pZ + Bb], axis=0)
            values = np.concatenate([Ca[cur], pC], axis=0)
            pC, pZ = Cb[cur], Zb[cur]
        else:
            logits = Za[cur] + Ba
            values = Ca[cur]
        S = _softmax_over_positions(logits)
        out[i] = np.sum(S * values, axis=0)
    return out


def overlap_transform(x: np.ndarray, pad_value: float) -> np.ndarray:
    """The Attention-evolution page's overlap transform (§3.1), without the batch
    axis: x [G, m, 2d] -> [G, 2m, d]; rows m..2m-1 take the current group's upper
    d channels, rows 0..m-1 the previous group's lower d channels, and the first
    group's history rows hold pad_value."""
    G, m, two_d = x.shape
    d = two_d // 2
    out = np.full((G, 2 * m, d), pad_value, dtype=np.float64)
    out[:, m:, :] = x[:, :, d:]
    out[1:, :m, :] = x[:-1, :, :d]
    return out


def compress_overlap_transform(kv, gate, ape, m: int) -> np.ndarray:
    """Overlapping compressor in the Attention-evolution page's formulation (§3.1):
    both the KV path and the gate path (logits + APE) go through the overlap
    transform (pads 0 and -inf), then a softmax over the 2m rows per channel and a
    weighted sum.  kv, gate: [n, 2d]; ape: [m, 2d]."""
    kv = np.asarray(kv, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    ape = np.asarray(ape, dtype=np.float64)
    n, two_d = kv.shape
    G = n // m
    kv_o = overlap_transform(kv.reshape(G, m, two_d), 0.0)
    lg_o = overlap_transform(gate.reshape(G, m, two_d) + ape[None], NEG_INF)
    out = np.empty((G, two_d // 2))
    for g in range(G):
        S = _softmax_over_positions(lg_o[g])
        out[g] = np.sum(S * kv_o[g], axis=0)
    return out


# =============================================================================
# RMSNorm and partial RoPE
# (DSA-to-CSA/HCA page, §Shared-KV MQA: RMSNorm on every query head and on the
# single compressed-KV head, RoPE on the last 64 dims, inverse rotation of the
# output by the query position; Attention-evolution page §4.1: kv_norm)
# =============================================================================

def rms_norm(x, eps: float = RMS_EPS) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope_cos_sin(pos: int, base: float = ROPE_BASE, n_rot: int = ROPE_DIMS):
    """cos/sin of pos * theta_j, theta_j = base^(-2j/n_rot), j < n_rot/2, in f64."""
    j = np.arange(n_rot // 2, dtype=np.float64)
    theta = base ** (-2.0 * j / n_rot)
    ang = np.fmod(float(pos) * theta, 2.0 * math.pi)
    return np.cos(ang), np.sin(ang)


def rope(x, pos: int, inverse: bool = False, base: float = ROPE_BASE) -> np.ndarray:
    """Rotate the last 64 dims of x (interleaved pairs) by +pos (or -pos)."""
    x = np.array(x, dtype=np.float64, copy=True)
    c = x.shape[-1]
    cos, sin = rope_cos_sin(pos, base)
    if inverse:
        sin = -sin
    x0 = x[..., c - ROPE_DIMS::2].copy()
    x1 = x[..., c - ROPE_DIMS + 1::2].copy()
    x[..., c - ROPE_DIMS::2] = x0 * cos - x1 * sin
    x[..., c - ROPE_DIMS + 1::2] = x0 * sin + x1 * cos
    return x


def compress_write(E, flags: int, m: int, pos0: int = 0, base: float = ROPE_BASE):
    """Write epilogue of the compressor: [RMSNorm] -> [RoPE at pos0 + m*i] ->
    [FP4 pack].  (Attention-evolution page §4.1: kv_norm after pooling; main KV
    then gets its position encoding and quantisation.)"""
    E = np.asarray(E, dtype=np.float64)
    if flags & NORM_W:
        E = rms_norm(E)
    if flags & ROPE_W:
        E = np.stack([rope(E[i], pos0 + m * i, base=base) for i in range(E.shape[0])]) \
            if E.shape[0] else E
    if flags & PACK_W:
        return nvfp4_pack(E.astype(np.float32))
    return E


# =============================================================================
# Lightning indexer, visibility, top-k, block pool
# =============================================================================

def visible_entries(t: int, m: int) -> int:
    """Entry j is visible to query t iff t >= m(j+1) (DSA-to-CSA/HCA page,
    §因果边界与短滑窗), so floor(t/m) entries are visible."""
    return t // m


def index_score(qI, w, KI, n_visible: int) -> np.ndarray:
    """I[s] = sum_h w[h] * ReLU(q^I_h . K^I_s) for s < n_visible, -inf beyond
    (DSA-to-CSA/HCA page eq. 16: no scale factor, no softmax).
    qI [H_I, d], w [H_I], KI [N, d]."""
    qI = np.asarray(qI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    KI = np.asarray(KI, dtype=np.float64)
    out = np.full(KI.shape[0], NEG_INF)
    V = int(n_visible)
    if V > 0:
        dots = KI[:V] @ qI.T                                   # [V, H_I]
        out[:V] = np.sum(w[None, :] * np.maximum(dots, 0.0), axis=1)
    return out


def _rank_order(values: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Positions of (values, ids) sorted by value descending, then id ascending."""
    return np.lexsort((ids, -values))


def topk(scores, n_visible: int, k: int) -> np.ndarray:
    """Top-k visible entries (DSA-to-CSA/HCA page eq. 17) by (score desc, index
    asc); if n_visible <= k all visible entries are returned.  Output: entry ids
    ascending, padded with -1 to length k."""
    s = np.asarray(scores, dtype=np.float64)[: int(n_visible)]
    ids = np.arange(s.shape[0])
    sel = np.sort(ids[_rank_order(s, ids)[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[: sel.shape[0]] = sel
    return out


def block_max(scores, n_visible: int, block: int = 8) -> np.ndarray:
    """Block score = max over the visible members of each block of `block`
    positions (CSA2 page, §解码器里的分层索引)."""
    s = np.asarray(scores, dtype=np.float64)
    V = int(n_visible)
    nb = (V + block - 1) // block
    return np.array([np.max(s[b * block: min(b * block + block, V)]) for b in range(nb)])


def block_pool(bmax, n_visible: int, block: int = 8, n_keep: int = 2048) -> np.ndarray:
    """Candidate pool of the hierarchical sparse indexer (CSA2 page,
    §解码器里的分层索引; Attention-evolution page §4.4): the newest visible block
    floor((V-1)/block) is always kept, the other n_keep-1 slots go to the best
    blocks by (block max desc, block asc).  Output ascending, -1 padded."""
    V = int(n_visible)
    out = np.full(n_keep, -1, dtype=np.int64)
    if V <= 0:
        return out
    nb = (V + block - 1) // block
    b_new = (V - 1) // block
    if nb <= n_keep:
        out[:nb] = np.arange(nb)
        return out
    bm = np.asarray(bmax, dtype=np.float64)[:nb]
    others = np.array([b for b in range(nb) if b != b_new])
    best = others[_rank_order(bm[others], others)[: n_keep - 1]]
    out[:] = np.sort(np.concatenate([best, [b_new]]))
    return out


def pool_candidates(pool_blocks, n_visible: int, block: int = 8) -> np.ndarray:
    """Entry ids covered by the pool's blocks that are visible, ascending."""
    ids = []
    for b in np.asarray(pool_blocks):
        if b < 0:
            continue
        for r in range(block):
            s = int(b) * block + r
            if s < n_visible:
                ids.append(s)
    return np.array(sorted(ids), dtype=np.int64)


def reindex_topk(full_scores, pool_blocks, n_visible: int, k: int, block: int = 8) -> np.ndarray:
    """Reindex layer selection in the 'official minimal' form (Attention-evolution
    page §4.4): full scores, then a candidate mask built from the pool, then top-k
    among the candidates by (score desc, index asc).  Output ascending, -1 padded."""
    cand = pool_candidates(pool_blocks, n_visible, block)
    s = np.asarray(full_scores, dtype=np.float64)[cand]
    sel = np.sort(cand[_rank_order(s, cand)[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[: sel.shape[0]] = sel
    return out


# =============================================================================
# Shared-KV MQA with window, sink, RMSNorm and partial RoPE
# (DSA-to-CSA/HCA page eqs. 18-19, eq. 27, §因果边界与短滑窗, and the page's
# sparse_shared_kv example; CSA2 page §保留了 CSA 的骨架: 512 selected entries plus
# the 128 most recent tokens' window)
# =============================================================================

def gather_keys(kv_entries, idx, swa, swa_pos0: int, t: int, window: int) -> np.ndarray:
    """Key/value rows for query t: the selected entries (id -1 skipped) followed by
    the window rows at positions max(0, t-window+1)..t; window slot of position p
    is (p - swa_pos0) mod cap."""
    rows = [np.asarray(kv_entries[int(s)], dtype=np.float64) for s in np.asarray(idx) if s >= 0]
    if window > 0:
        cap = swa.shape[0]
        for p in range(max(0, t - window + 1), t + 1):
            rows.append(np.asarray(swa[(p - swa_pos0) % cap], dtype=np.float64))
    c = np.asarray(kv_entries).shape[-1] if len(rows) == 0 else rows[0].shape[0]
    return np.array(rows, dtype=np.float64).reshape(len(rows), c)


def attend(q, keys, t: int, sink=None, flags: int = QNORM | KVNORM | ROPE,
           base: float = ROPE_BASE) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Core attention of one query over given key/value rows, all heads.

    q [H, c]; keys [nk, c] (each row is both key and value).  Steps: q^ =
    RoPE_t(RMSNorm(q)); k^_j = RMSNorm(row_j); z_j = q^ . k^_j / sqrt(c);
    p_j = e^{z_j} / (sum_l e^{z_l} + e^{sink_h}) (eq. 27; sink None = no sink term);
    o = RoPE_{-t}(sum_j p_j k^_j).  Returns (o [H, c], lse [H], mass [H]) with
    lse = log(sum_j e^{z_j} + e^{sink_h})."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(keys, dtype=np.float64)
    H, c = q.shape
    if flags & KVNORM and K.shape[0]:
        K = rms_norm(K)
    qh = rms_norm(q) if flags & QNORM else q
    if flags & ROPE:
        qh = rope(qh, t, base=base)
    z = qh @ K.T / math.sqrt(c)                                  # [H, nk]
    s = np.full(H, NEG_INF) if sink is None else np.asarray(sink, dtype=np.float64)
    mx = np.maximum(np.max(z, axis=1) if K.shape[0] else np.full(H, NEG_INF), s)
    ez = np.exp(z - mx[:, None])
    denom = np.sum(ez, axis=1) + np.exp(s - mx)
    p = ez / denom[:, None]
    o = p @ K
    if flags & ROPE:
        o = rope(o, t, inverse=True, base=base)
    lse = mx + np.log(denom)
    return o, lse, np.sum(p, axis=1)


def sparse_attn(q, kv_entries, idx, swa, swa_pos0: int, t: int, sink=None, window: int = 128,
                flags: int = QNORM | KVNORM | ROPE, base: float = ROPE_BASE):
    keys = gather_keys(kv_entries, idx, swa, swa_pos0, t, window)
    return attend(q, keys, t, sink, flags, base)


# =============================================================================
# Whole-layer helpers (loops over batch and queries)
# =============================================================================

def dense_attn(q, kv_entries, swa, swa_pos0: int, t: int, m: int, sink=None, window: int = 128,
               flags: int = QNORM | KVNORM | ROPE, base: float = ROPE_BASE):
    """HCA attention (DSA-to-CSA/HCA page «HCA：公式 (20)–(26)», eq. 26): every compressed
    entry visible to query t (floor(t/m) of them, m = m' = 128 in V4) is key and
    value, together with the window (section «因果边界与短滑窗»).  The selection step
    of CSA is simply absent, so this is sparse_attn with the index list 0..V-1."""
    V = visible_entries(int(t), m)
    idx = np.arange(V, dtype=np.int64)
    return sparse_attn(q, kv_entries, idx, swa, swa_pos0, t, sink, window, flags, base)


def full_layer_decode(qI, w, KI, q, kv_entries, swa, swa_pos0, q_pos, m, sink, k=512,
                      window=128, use_pool=False, block=8, n_keep=2048, flags=QNORM | KVNORM | ROPE):
    """One Full-mode layer for the queries of one sequence: score, [pool], top-k,
    attention.  qI [Q, H_I, d], w [Q, H_I], KI [N, d], q [Q, H, c]."""
    res = []
    for i, t in enumerate(np.asarray(q_pos)):
        V = visible_entries(int(t), m)
        sc = index_score(qI[i], w[i], KI, V)
        idx = topk(sc, V, k)
        pool = block_pool(block_max(sc, V, block), V, block, n_keep) if use_pool else None
        o, lse, mass = sparse_attn(q[i], kv_entries, idx, swa, swa_pos0, int(t), sink, window, flags)
        res.append(dict(scores=sc, idx=idx, pool=pool, out=o, lse=lse, mass=mass))
    return res


# =============================================================================
# Sharding one long sequence over P ranks (entry ranges): exact merges
# =============================================================================

def merge_topk(rank_ids, rank_scores, k: int) -> np.ndarray:
    """Merge per-rank top-k lists (global entry ids and their scores) into the
    global top-k by (score desc, id asc); ascending output, -1 padded."""
    ids = np.concatenate([np.asarray(r, dtype=np.int64) for r in rank_ids])
    sc = np.concatenate([np.asarray(r, dtype=np.float64) for r in rank_scores])
    keep = ids >= 0
    ids, sc = ids[keep], sc[keep]
    sel = np.sort(ids[_rank_order(sc, ids)[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[: sel.shape[0]] = sel
    return out


def merge_attn(parts_o, parts_lse, sink=None):
    """Combine partial attention results computed without the sink over disjoint
    key sets: o = sum_r e^{lse_r - L} o_r with L = log(sum_r e^{lse_r} + e^{sink})."""
    lses = np.stack([np.asarray(l, dtype=np.float64) for l in parts_lse])      # [P, H]
    os_ = np.stack([np.asarray(o, dtype=np.float64) for o in parts_o])         # [P, H, c]
    s = np.full(lses.shape[1], NEG_INF) if sink is None else np.asarray(sink, dtype=np.float64)
    mx = np.maximum(np.max(lses, axis=0), s)
    denom = np.sum(np.exp(lses - mx), axis=0) + np.exp(s - mx)
    L = mx + np.log(denom)
    wts = np.exp(lses - L)                                                     # [P, H]
    return np.sum(wts[:, :, None] * os_, axis=0), L
