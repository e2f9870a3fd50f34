// mask.cuh - element masks as per-row (or per-key) index intervals, the
// classification of a 128 x 128 kernel tile, and the walk over block-sparse
// lists shared by every attention kernel.
//
// Mask kinds follow "Enable 2CTA for SM100 block-sparse backward" (fuzz
// tester mask names: causal, sliding_window, block_diagonal, mini_causal,
// prefix_lm; mini_causal, which the page does not define, is read as causal
// inside each block of block_size keys) and
// the dynamic (bias-ranked) mask of "Optimize Flash Dynamic Mask Attention
// Kernel Configurations". With the diagonal aligned bottom-right
// (a = i + Sk - Sq), every closed-form kind allows, for query i, one interval
// of keys [lo_i, hi_i]; lo_i and hi_i never decrease with i. The dynamic kind
// is the causal interval intersected with a per-(b,h) keep bitmask.
//
// Gathered keys (dynamic kind with the kept-key index list): the kernels
// stream only the kept keys, in ascending index order, as compact tiles.
// Compact key c stands for key pos[c]; query i sees compact keys
// [0, kept(<= i + Sk - Sq)), a prefix, so the tile classes and the element
// masks reduce to one count per query row (and one position per key).
#pragma once

#include "common.cuh"

namespace gb {

struct MaskParams {
  int kind;
  int window_left;
  int block_size;
  int prefix_len;
  float slope;             // rel-bias slope (score += slope * (i - j))
  const float* key_bias;   // [B*H, Sk] or nullptr
  const uint32_t* keep;    // [B*H, nkw] (dynamic) or nullptr
  int nkw;                 // words per (b,h) in keep; words per row of table
  const uint32_t* table;   // element table: [Sq, nkw] or [B*H, Sq, nkw] bits, or nullptr
  int table_per_head;      // 1: one table per (b, h)
};

// Row i's words of the element table (mask kind TABLE) of head bh.
__device__ __forceinline__ const uint32_t* table_row(const MaskParams& m, int bh, int Sq, int i) {
  return m.table + ((m.table_per_head ? (size_t)bh * Sq : 0) + (size_t)i) * m.nkw;
}

// ---- gathered keys ----------------------------------------------------------
// Number of kept keys with index <= a among the keep bits of one head (nkw
// words); warp-collective (every lane gets the count), a warp-uniform.
__device__ __forceinline__ int warp_kept_upto(const uint32_t* keep, int nkw, int a) {
  if (a < 0) return 0;
  const int lane = threadIdx.x & 31;
  const int wa = min(a >> 5, nkw - 1);
  const uint32_t last = (a >> 5) > wa ? 0xffffffffu : ((2u << (a & 31)) - 1u);
  int cnt = 0;
#pragma unroll 4
  for (int w = lane; w <= wa; w += 32) {
    const uint32_t b = __ldg(keep + w);
    cnt += __popc(w == wa ? (b & last) : b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt;
}

// Kept keys with index in [lo, hi] (a short range: a few words).
__device__ __forceinline__ int kept_between(const uint32_t* keep, int nkw, int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, nkw * 32 - 1);
  int cnt = 0;
  for (int w = lo >> 5; w <= (hi >> 5); ++w) {
    uint32_t b = __ldg(keep + w);
    const int wb = w << 5;
    if (lo > wb) b &= ~((1u << (lo - wb)) - 1u);
    if (hi < wb + 31) b &= (2u << (hi - wb)) - 1u;
    cnt += __popc(b);
  }
  return cnt;
}

// Compact-key count seen by each query row of a warp (32 consecutive rows
// i0 + lane, i.e. positions a0 + lane with a0 = i0 + Sk - Sq): returns the
// lane's last visible compact key (count - 1; -1 when none). Warp-collective.
__device__ __forceinline__ int gathered_row_hi(const uint32_t* keep, int nkw, int a0) {
  const int lane = threadIdx.x & 31;
  const int base = warp_kept_upto(keep, nkw, a0 - 1);
  const int a = a0 + lane;
  const int extra = a < 0 ? 0 : kept_between(keep, nkw, max(a0, 0), a);
  return base + extra - 1;
}

// Forward direction (fixed 128-row query tile, streamed compact key tiles):
// c_first / c_last = compact keys visible to the tile's first / last row.
__device__ __forceinline__ bool gathered_slot_rows(int s, int c_first, int c_last, int* start, bool* masked) {
  const int st = s * 128;
  if (st >= c_last) return false;
  *start = st;
  *masked = st + 128 > c_first;
  return true;
}

// Backward direction (fixed compact key tile, streamed 128-row query tiles):
// p_first / p_last = original index of the tile's first / last key; kfull =
// the key tile has 128 keys; delta = Sk - Sq. Query i sees key p iff
// p <= i + delta.
__device__ __forceinline__ bool gathered_slot_cols(int s, int p_first, int p_last, bool kfull, int delta, int Sq,
                                                   int* start, bool* masked) {
  const int st = s * 128;
  const int q1 = min(st + 128, Sq);
  if (st >= Sq || p_first > q1 - 1 + delta) return false;
  *start = st;
  *masked = !(kfull && q1 - st == 128 && p_last <= st + delta);
  return true;
}

// Allowed keys of query i: [lo, hi] (inclusive, clipped to [0, Sk-1]);
// empty when lo > hi.
__device__ __forceinline__ void row_interval(const MaskParams& m, int i, int Sq, int Sk, int& lo, int& hi) {
  const int a = i + (Sk - Sq);
  lo = 0;
  hi = Sk - 1;
  switch (m.kind) {
    case GBATTN_MASK_CAUSAL:
    case GBATTN_MASK_DYNAMIC_TOPK:
      hi = min(a, Sk - 1);
      break;
    case GBATTN_MASK_SLIDING:
      hi = min(a, Sk - 1);
      if (m.window_left >= 0) lo = max(0, a - m.window_left);
      break;
    case GBATTN_MASK_BLOCK_DIAG: {
      const int blk = floor_div(a, m.block_size) * m.block_size;
      lo = max(0, blk);
      hi = min(Sk - 1, blk + m.block_size - 1);
      break;
    }
    case GBATTN_MASK_MINI_CAUSAL: {
      const int blk = floor_div(a, m.block_size) * m.block_size;
      lo = max(0, blk);
      hi = min(Sk - 1, a);
      break;
    }
    case GBATTN_MASK_PREFIX_LM:
      hi = min(max(m.prefix_len - 1, a), Sk - 1);
      break;
    default:
      break;
  }
}

// Queries that may see key j: [lo, hi] (inclusive, clipped to [0, Sq-1]);
// the transpose of row_interval (ignores the dynamic keep bit, which the
// caller tests separately).
__device__ __forceinline__ void col_interval(const MaskParams& m, int j, int Sq, int Sk, int& lo, int& hi) {
  const int d = Sk - Sq;  // a = i + d
  lo = 0;
  hi = Sq - 1;
  switch (m.kind) {
    case GBATTN_MASK_CAUSAL:
    case GBATTN_MASK_DYNAMIC_TOPK:
      lo = max(0, j - d);
      break;
    case GBATTN_MASK_SLIDING:
      lo = max(0, j - d);
      if (m.window_left >= 0) hi = min(Sq - 1, j - d + m.window_left);
      break;
    case GBATTN_MASK_BLOCK_DIAG: {
      const int blk = floor_div(j, m.block_size) * m.block_size;
      lo = max(0, blk - d);
      hi = min(Sq - 1, blk + m.block_size - 1 - d);
      break;
    }
    case GBATTN_MASK_MINI_CAUSAL: {  // rows with j <= i + d inside key j's block
      const int blk = floor_div(j, m.block_size) * m.block_size;
      lo = max(0, j - d);
      hi = min(Sq - 1, blk + m.block_size - 1 - d);
      break;
    }
    case GBATTN_MASK_PREFIX_LM:
      if (j >= m.prefix_len) lo = max(0, j - d);
      break;
    default:
      break;
  }
}

enum { TILE_EMPTY = 0, TILE_PARTIAL = 1, TILE_FULL = 2 };

// Class of the tile rows [q0, q0+128) x keys [k0, k0+128), rows clipped to
// Sq and keys to Sk. EMPTY is exact when returned (no allowed pair); FULL
// is exact when returned (every pair allowed, nothing clipped, and - when
// rows_whole - no padding row); otherwise PARTIAL (element masks applied).
__device__ __forceinline__ int tile_class(const MaskParams& m, int q0, int k0, int Sq, int Sk,
                                          bool rows_whole) {
  const int q1 = min(q0 + 128, Sq);
  const int k1 = min(k0 + 128, Sk);
  if (q1 <= q0 || k1 <= k0) return TILE_EMPTY;
  int lo_f, hi_f, lo_l, hi_l;
  row_interval(m, q0, Sq, Sk, lo_f, hi_f);
  row_interval(m, q1 - 1, Sq, Sk, lo_l, hi_l);
  if (hi_l < k0 || lo_f > k1 - 1) return TILE_EMPTY;
  if (m.kind == GBATTN_MASK_DYNAMIC_TOPK || m.kind == GBATTN_MASK_TABLE) return TILE_PARTIAL;
  const bool whole = (k1 - k0 == 128) && (!rows_whole || q1 - q0 == 128);
  if (whole && lo_l <= k0 && hi_f >= k1 - 1) return TILE_FULL;
  return TILE_PARTIAL;
}

// Walk over the 128-wide tiles a CTA streams. The CTA owns a fixed 128-range
// of the other dimension; the lists (mask list first, then full list) name
// sparse blocks of `span` = (sub * 128) positions along the streamed
// dimension. Slot s = (list entry) * sub + (sub-tile). Every role of a CTA
// walks the same slots and keeps the same ones, so they agree on the order.
struct TileWalk {
  const int32_t* mlist;  // mask-list entries of this CTA's block row
  const int32_t* flist;  // full-list entries
  int mcnt, fcnt;
  int sub;               // sub-tiles per sparse block
  int nblk;              // number of sparse blocks along the streamed dim
  int limit;             // Sk (forward) or Sq (backward)
  int nslots;
};

// Returns false for a slot that is skipped (beyond the sequence end, empty
// sub-tile, or a corrupt list entry, which also raises GBATTN_ERR_BLOCKS).
// On true, *start is the first streamed index and *masked says whether the
// element mask must be applied.
__device__ __forceinline__ bool walk_slot(const TileWalk& w, int s, const MaskParams& m, bool forward,
                                          int fixed0, int Sq, int Sk, int* start, bool* masked) {
  const int e = s / w.sub;
  const int u = s - e * w.sub;
  const bool from_mask = e < w.mcnt;
  const int blk = from_mask ? __ldg(w.mlist + e) : __ldg(w.flist + (e - w.mcnt));
  if (blk < 0 || blk >= w.nblk) {
    if (u == 0) raise_dev_error(GBATTN_ERR_BLOCKS);
    return false;
  }
  const int st = (blk * w.sub + u) * 128;
  if (st >= w.limit) return false;
  *start = st;
  if (!from_mask) {
    *masked = false;
    return true;
  }
  const int cls = forward ? tile_class(m, fixed0, st, Sq, Sk, false) : tile_class(m, st, fixed0, Sq, Sk, true);
  if (cls == TILE_EMPTY) return false;
  *masked = (cls != TILE_FULL);
  return true;
}

__device__ __forceinline__ TileWalk make_walk(const int32_t* mcnt, const int32_t* midx, const int32_t* fcnt,
                                              const int32_t* fidx, int row, int nblk, int sub, int limit) {
  TileWalk w;
  int mc = __ldg(mcnt + row);
  int fc = __ldg(fcnt + row);
  if (mc < 0 || mc > nblk || fc < 0 || fc > nblk || mc + fc > nblk) {
    raise_dev_error(GBATTN_ERR_BLOCKS);
    mc = 0;
    fc = 0;
  }
  w.mlist = midx + (size_t)row * nblk;
  w.flist = fidx + (size_t)row * nblk;
  w.mcnt = mc;
  w.fcnt = fc;
  w.sub = sub;
  w.nblk = nblk;
  w.limit = limit;
  w.nslots = (mc + fc) * sub;
  return w;
}

// Dense walk (no lists, mask kind NONE): every 128-tile of [0, limit).
__device__ __forceinline__ bool dense_slot(int s, const MaskParams& m, bool forward, int fixed0, int Sq,
                                           int Sk, int* start, bool* masked) {
  const int st = s * 128;
  const int cls = forward ? tile_class(m, fixed0, st, Sq, Sk, false) : tile_class(m, st, fixed0, Sq, Sk, true);
  if (cls == TILE_EMPTY) return false;
  *start = st;
  *masked = (cls != TILE_FULL);
  return true;
}

// The visited tiles of a CTA, computed once into shared memory by one warp
// (32 slots at a time, compacted in slot order), so that every role reads its
// next tile with one shared load. Entry = (start / 128) << 1 | masked. If a
// CTA visits more than `cap` tiles the roles walk the slots themselves.
template <class SlotFn>
__device__ __forceinline__ void build_tile_list(SlotFn slot, int nslots, uint16_t* list, int cap, int* count) {
  const int lane = threadIdx.x & 31;
  int cnt = 0;
  for (int s0 = 0; s0 < nslots; s0 += 32) {
    const int s = s0 + lane;
    int st = 0;
    bool mk = false;
    const bool v = (s < nslots) && slot(s, &st, &mk);
    const unsigned b = __ballot_sync(0xffffffffu, v);
    const int pos = cnt + __popc(b & ((1u << lane) - 1u));
    if (v && pos < cap) list[pos] = (uint16_t)(((st >> 7) << 1) | (mk ? 1 : 0));
    cnt += __popc(b);
  }
  if (lane == 0) *count = cnt;
}

template <class SlotFn>
struct TileSeq {
  const uint16_t* list;
  int count, use_list, nslots, s, t;
  SlotFn slot;
  __device__ __forceinline__ bool next(int* start, bool* masked) {
    if (use_list) {
      if (t >= count) return false;
      const uint32_t e = list[t++];
      *start = (int)(e >> 1) * 128;
      *masked = (e & 1u) != 0;
      return true;
    }
    while (s < nslots) {
      if (slot(s++, start, masked)) return true;
    }
    return false;
  }
};
template <class SlotFn>
__device__ __forceinline__ TileSeq<SlotFn> tile_seq(SlotFn slot, const uint16_t* list, int count, int cap,
                                                    int nslots) {
  return TileSeq<SlotFn>{list, count, count <= cap ? 1 : 0, nslots, 0, 0, slot};
}

// Per-key score terms (key bias_j - slope * j) * log2(e) of one warp's 64
// key columns [cb, cb + 64) of each visited tile, j the key's original index
// (pos[] of the compact index for gathered keys). With a key bias the loads
// run ahead of the tiles: while tile n is processed, the original indices of
// tile n + 2 and the bias values of tile n + 1 are loaded, so the dependent
// index -> bias loads never stall the caller. `seq` must be a copy of the
// caller's tile sequence taken before its first next().
template <bool GAT, class Seq, int NV = 2>
struct KeyTerms {
  Seq ahead;
  const float* kb;   // key bias of this head, or nullptr
  const int32_t* pos;  // gathered keys: original index of each compact key
  int skv, col0;       // streamed key extent; col0 = cb + lane
  float slope;
  int jo_cur[NV], jo_nx[NV];
  float bv_cur[NV];

  __device__ __forceinline__ int key_of(int st, int e) const {
    const int j = st + col0 + e * 32;
    if (j >= skv) return -1;
    if constexpr (GAT) return __ldg(pos + j);
    return j;
  }
  __device__ __forceinline__ void start() {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      jo_cur[e] = jo_nx[e] = -1;
      bv_cur[e] = 0.f;
    }
    if (!kb) return;
    int st;
    bool mk;
    if (ahead.next(&st, &mk)) {
#pragma unroll
      for (int e = 0; e < NV; ++e) jo_cur[e] = key_of(st, e);
    }
#pragma unroll
    for (int e = 0; e < NV; ++e) bv_cur[e] = jo_cur[e] >= 0 ? __ldg(kb + jo_cur[e]) : 0.f;
    if (ahead.next(&st, &mk)) {
#pragma unroll
      for (int e = 0; e < NV; ++e) jo_nx[e] = key_of(st, e);
    }
  }
  // Writes this lane's two terms of the tile starting at compact key kv0
  // (the tile the caller's sequence just returned) to ct[lane], ct[32 + lane].
  __device__ __forceinline__ void emit(int kv0, float* ct) {
    if (kb) {
#pragma unroll
      for (int e = 0; e < NV; ++e)
        ct[e * 32 + (col0 & 31)] = jo_cur[e] >= 0 ? (bv_cur[e] - slope * (float)jo_cur[e]) * kLog2e : 0.f;
      int st;
      bool mk;
      int jo_n2[NV];
#pragma unroll
      for (int e = 0; e < NV; ++e) jo_n2[e] = -1;
      if (ahead.next(&st, &mk)) {
#pragma unroll
        for (int e = 0; e < NV; ++e) jo_n2[e] = key_of(st, e);
      }
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        bv_cur[e] = jo_nx[e] >= 0 ? __ldg(kb + jo_nx[e]) : 0.f;
        jo_cur[e] = jo_nx[e];
        jo_nx[e] = jo_n2[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int jo = key_of(kv0, e);
        ct[e * 32 + (col0 & 31)] = jo >= 0 ? -slope * (float)jo * kLog2e : 0.f;
      }
    }
  }
};
// The same terms loaded when each tile starts (no look-ahead state).
struct KeyTermsDirect {
  const float* kb;
  int skv, col0;
  float slope;
  __device__ __forceinline__ void emit(int kv0, float* ct) const {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = kv0 + col0 + e * 32;
      ct[e * 32 + (col0 & 31)] = j < skv ? ((kb ? __ldg(kb + j) : 0.f) - slope * (float)j) * kLog2e : 0.f;
    }
  }
};
template <bool GAT, int NV = 2, class Seq>
__device__ __forceinline__ KeyTerms<GAT, Seq, NV> key_terms(const Seq& seq, const float* kb, const int32_t* pos,
                                                           int skv, int col0, float slope) {
  KeyTerms<GAT, Seq, NV> t{seq, kb, pos, skv, col0, slope, {}, {}, {}};
  t.start();
  return t;
}

}  // namespace gb
