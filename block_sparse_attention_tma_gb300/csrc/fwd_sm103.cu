// fwd_sm103.cu - fused attention forward on the 5th-generation tensor cores.
//
// Method: "Optimize Flash Dynamic Mask Attention Kernel Configurations"
// (forward kernel; masks, softcap) and "Enable 2CTA for SM100 block-sparse
// backward" (forward driven by block-sparse lists, q/kv sub-tiling of a
// sparse block into 128 x 128 kernel tiles, QK/V head dims 192/128). The
// running max / sum update is the online-softmax merge of the POPCORNBENCH
// "Kimi-K2.6 l1_p97" trace (m_new = max, rescale by exp(m_old - m_new)).
//
// One CTA = one (b, h, 128-row query tile); 10 warps:
//   warp 0      TMA producer: Q once, then K and V tiles into rings.
//   warp 1      MMA issuer (one thread): S = Q K^T with Q read from TMEM
//               (A operand) and K from shared memory, into one of two TMEM S
//               buffers; O += P V with P read from TMEM and V (MN-major) from
//               shared memory.
//   warps 2..9  softmax, two warps per TMEM lane quarter: thread = (query
//               row, half of the 128 key columns). Group 0 copies the Q rows
//               into TMEM once. Per tile each thread loads its 64 S values,
//               masks (partial tiles only), folds scale * log2(e) and the
//               per-key bias term into one FMA, exchanges its partial row max
//               with the other half through shared memory (the two warps of a
//               lane quarter meet at a named barrier per tile), exp2, writes its
//               half of P (bf16) back over the S buffer, and rescales its half
//               of O only when the row max grows by more than 2^8 ("lazy"
//               rescale); final O / l and LSE. Two warps per SM sub-partition
//               hide the latencies one warp alone cannot.
// Keeping Q in TMEM means the QK^T MMA reads only K from shared memory; the
// shared-memory traffic per tile (K + V reads, K + V TMA writes) then fits
// the time of the two MMAs.
// Gathered keys (dynamic top-k mask with its kept-key index list): the key
// tiles are compact tiles of kept keys only, which the producer warp copies
// row by row with 16-byte cp.async into the swizzled tile layout (completion
// tracked on the tile's mbarrier); the bias and rel-bias terms use each key's
// original index, loaded a tile ahead, and the element mask is the prefix of
// compact keys each row sees. No key outside the keep set is loaded or
// multiplied.
// Packed decode (grouped-query attention, split-KV): the G x Sq query rows of
// a key/value head (contiguous in Q and O) form the 128-row tiles, so one CTA
// streams each key/value tile once for the whole group and the tensor cores
// take the score and output products; a CTA covers one split of the keys and
// writes a normalised partial output and LSE that the split combine merges.
// Softmax warps whose rows hold no query row of the group only keep the
// barriers in step.
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+Dv), Q [384, 384+Dqk/2).
#include "kernels.h"
#include "mask.cuh"

namespace gb {

// 64 TMEM columns in one load (32 lanes x 64 x 32 bit); the softmax warps'
// S tile half (the backward kernels keep two 32-column loads: with this one
// their gathered / softcap variants spill and they measured no faster).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : GB_R16(r, 0), GB_R16(r, 16), GB_R16(r, 32), GB_R16(r, 48)
      : "r"(taddr));
}

// Named barrier `id` (1..15; 0 is __syncthreads) over `count` threads that
// also returns the OR of their predicates. Every participant must reach it:
// callers pass their failure flag through it and leave their loop together.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;
  int B, H, Sq, Sk;
  int Hkv, G;          // key/value heads and query heads per key/value head (GQA)
  int nqt;             // query tiles per head
  float scale_log2;    // scale * log2(e)
  float cap_pre;       // scale / softcap (softcap on)
  float cap_post;      // softcap * log2(e)
  MaskParams mask;
  int has_lists;
  int gather;          // gathered keys: rows of gk / gv copied by index
  int Skv;             // streamed key extent (Sk, or the kept-key count)
  const int32_t* kidx; // [B*H, Sk] kept key indices (gathered keys)
  const __nv_bfloat16 *gk, *gv;  // K [B*H*Sk, Dqk], V [B*H*Sk, Dv] (gathered keys)
  int sub;             // sparse_n / 128
  int hgroup;          // CTA order: heads per group (head_group), 0 = none
  int nqb, nkb, sparse_m;
  const int32_t *mcnt, *midx, *fcnt, *fidx;  // forward lists
  __nv_bfloat16* o;
  float* lse;
  // packed decode: rows per group, row tiles per group, splits, keys per split
  int pk_R, pk_nrt, pk_nsplit;
  float *o_part, *lse_part;  // [nsplit][B*H*Sq][Dv], [nsplit][B*H*Sq] (nsplit > 1)
  const int32_t* pk_seqlens;  // [B] keys per sequence, or nullptr (all Sk)
  const int32_t* pk_pages;    // [B][pk_max_pages] page table, or nullptr (dense cache):
                              // tm_k / tm_v then map the pool [num_pages * Hkv, page_size, D]
  int pk_page_size, pk_max_pages, pk_num_pages;
  unsigned long long wait_ns;  // time limit of every wait (0 = kWaitLimitNs)
  int test_withhold_k;         // test hook: the K tile of the first visited tile is never loaded
};

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int SWQ = DQK >= 64 ? 128 : 64;  // swizzle span of Q/K rows
  static constexpr int SWV = DV >= 64 ? 128 : 64;
  static constexpr int QSLAB = 128 * SWQ;           // bytes of one 128-row slab
  static constexpr int NQSLAB = DQK * 2 / SWQ;
  static constexpr int QTILE = 128 * DQK * 2;
  static constexpr int VSLAB = 128 * SWV;
  static constexpr int NVSLAB = DV * 2 / SWV;
  static constexpr int VTILE = 128 * DV * 2;
  static constexpr int KST = DQK >= 192 ? 2 : 3;
  static constexpr int VST = DQK >= 128 ? 2 : 3;
  static constexpr int T_O = 256, T_Q = 384;
  static_assert(T_Q + DQK / 2 <= 512 && T_O + DV <= T_Q, "TMEM budget");
  // barriers: q_full, q_tmem, k_full[KST], k_empty[KST], v_full[VST],
  // v_empty[VST], s_full[2], p_full[2], o_done, drain, fin, o_fin
  static constexpr int NBAR = 2 + 2 * KST + 2 * VST + 2 + 2 + 1 + 1 + 1 + 1;
  // softmax warps: NG per TMEM lane quarter, each thread one query row and
  // CWF = 128 / NG of the tile's key columns. NG = 4 (18 warps) caps a thread
  // at 96 registers and measured slower (16K causal MLA 1.091 -> 1.243 ms),
  // so every shape keeps two.
  static constexpr int NG = 2, CWF = 128 / NG;
  static constexpr int THREADS = 64 + 128 * NG;
  // + 4 KB tail slack; at least 120 KB so that one CTA holds an SM (its 512
  // TMEM columns are the whole TMEM)
  // colterm [4 NG warps][2][CWF] + row-max exchange [2][NG][128] + row sums [NG][128]
  static constexpr int TCAP = 1024;  // visited-tile list entries (uint16)
  static constexpr int SMEM_USED = 1024 + QTILE + KST * QTILE + VST * VTILE + 8 * 128 * 4 + 2 * NG * 128 * 4 +
                                   NG * 128 * 4 + TCAP * 2 + NBAR * 8 + 32 + 2048;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, DV, false, true);
};

// Loads 128 consecutive TMEM columns of this thread's lane into r[].
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t* r) {
  tmem_ld32(taddr + 0, r);
  tmem_ld32(taddr + 32, r + 32);
  tmem_ld32(taddr + 64, r + 64);
  tmem_ld32(taddr + 96, r + 96);
  tmem_wait_ld32(r);
  reg_fence32(r + 32);
  reg_fence32(r + 64);
  reg_fence32(r + 96);
}

template <int DQK, int DV, bool CAP, bool GAT, bool PK = false>
__global__ void __launch_bounds__(FwdCfg<DQK, DV>::THREADS, 1) fwd_bf16_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + C::QTILE;
  uint8_t* sV = sK + C::KST * C::QTILE;
float* colterm = reinterpret_cast<float*>(sV + C::VST * C::VTILE);  // [4 NG warps][2][CWF]
  float* xmax = colterm + 8 * 128;                                     // [2][NG column groups][128 rows]
  float* xsum = xmax + 2 * C::NG * 128;                                // [NG column groups][128 rows]
  uint16_t* tlist = reinterpret_cast<uint16_t*>(xsum + 2 * 128);  // [TCAP]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tlist + C::TCAP);
  uint64_t* q_full = bars;
  uint64_t* q_tmem = q_full + 1;
  uint64_t* k_full = q_tmem + 1;
  uint64_t* k_empty = k_full + C::KST;
  uint64_t* v_full = k_empty + C::KST;
  uint64_t* v_empty = v_full + C::VST;
  uint64_t* s_full = v_empty + C::VST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint64_t* fin = drain + 1;
  // one phase: every PV product of the CTA has completed (the epilogue's wait;
  // a parity wait on o_done there could pass two phases early)
  uint64_t* o_fin = fin + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(tmem_slot + 1), p.wait_ns);
  int* tcount = reinterpret_cast<int*>(tmem_slot + 2);
  int* gcount = reinterpret_cast<int*>(tmem_slot + 4);  // [2] gathered keys seen by the first / last row

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int L = blockIdx.x;
  int bh, bkv, q0;
  // packed decode: this CTA's keys [kbeg, kend), its rows' query positions
  // [pa, pb], its split and the row id of its group's first row
  int kbeg = 0, kend = p.Sk, pa = 0, pb = 0, split = 0, row_base = 0;
  int skb = p.Sk;  // keys of this sequence (packed decode with per-sequence counts)
  if constexpr (PK) {
    split = L % p.pk_nsplit;
    const int rest = L / p.pk_nsplit;
    const int rt = rest % p.pk_nrt;
    bkv = rest / p.pk_nrt;
    bh = (bkv / p.Hkv) * p.H + (bkv % p.Hkv) * p.G;  // first query head of the group
    row_base = bh * p.Sq;
    q0 = rt * 128;  // first group row of this CTA
    if (p.pk_seqlens) {
      skb = __ldg(p.pk_seqlens + bkv / p.Hkv);
      const int cap = p.pk_pages ? p.pk_max_pages * p.pk_page_size : p.Sk;
      if (skb < 0 || skb > cap) {
        if (threadIdx.x == 0) raise_dev_error(GBATTN_ERR_BLOCKS);
        skb = max(0, min(skb, cap));
      }
    }
    // split s covers keys [s L, (s + 1) L), L = ceil(keys / n) rounded up to 128
    const int per = ((skb + p.pk_nsplit - 1) / p.pk_nsplit + 127) / 128 * 128;
    kbeg = split * per;
    kend = min(kbeg + per, skb);
    const int r1 = min(q0 + 127, p.pk_R - 1);
    if (q0 / p.Sq == r1 / p.Sq) {
      pa = q0 % p.Sq;
      pb = r1 % p.Sq;
    } else {
      pa = 0;
      pb = p.Sq - 1;
    }
  } else {
    int t;
    grid_tile(L, BH, p.nqt, p.hgroup, &bh, &t);
    const int qt = p.nqt - 1 - t;  // heaviest (last) query tiles first
    bkv = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;  // key/value head of this query head
    q0 = qt * 128;
  }
  constexpr bool gat = GAT;  // gathered keys (compile-time: the list walk keeps its own code)
  const int Skv = PK ? skb : p.Skv;
  const int SkM = PK ? skb : p.Sk;  // key count the masks align to
  const int delta = p.Sk - p.Sq;
  const uint32_t* keep_h = p.mask.keep ? p.mask.keep + (size_t)bh * p.mask.nkw : nullptr;
  const int32_t* pos_h = gat ? p.kidx + (size_t)bh * p.Sk : nullptr;

  // Tile walk of this CTA; warp 0 compacts it into shared memory once.
  TileWalk walk;
  int nslots;
  int c_first = 0, c_last = 0;
  if (PK) {
    nslots = kend > kbeg ? (kend + 127) / 128 - kbeg / 128 : 0;
  } else if (gat) {
    nslots = (Skv + 127) / 128;
  } else if (p.has_lists) {
    const int r = q0 / p.sparse_m;
    walk = make_walk(p.mcnt, p.midx, p.fcnt, p.fidx, bh * p.nqb + r, p.nkb, p.sub, p.Sk);
    nslots = walk.nslots;
  } else {
    nslots = (p.Sk + 127) / 128;
  }
  auto slot = [&](int s, int* kv0, bool* masked) -> bool {
    if constexpr (PK) {
      // rows at query positions [pa, pb] (monotone intervals: the first and
      // last position bound every row's interval)
      const int st = kbeg + s * 128, k1 = min(st + 128, SkM);
      int lo_a, hi_a, lo_b, hi_b;
      row_interval(p.mask, pa, p.Sq, SkM, lo_a, hi_a);
      row_interval(p.mask, pb, p.Sq, SkM, lo_b, hi_b);
      if (hi_b < st || lo_a > k1 - 1) return false;
      *kv0 = st;
      *masked = !(k1 - st == 128 && lo_b <= st && hi_a >= k1 - 1);
      return true;
    }
    if (gat) return gathered_slot_rows(s, c_first, c_last, kv0, masked);
    return p.has_lists ? walk_slot(walk, s, p.mask, true, q0, p.Sq, p.Sk, kv0, masked)
                       : dense_slot(s, p.mask, true, q0, p.Sq, p.Sk, kv0, masked);
  };
  if (warp == 0) {
    if (gat) {
      c_first = warp_kept_upto(keep_h, p.mask.nkw, q0 + delta);
      c_last = warp_kept_upto(keep_h, p.mask.nkw, min(q0 + 127, p.Sq - 1) + delta);
      if (lane == 0) {
        gcount[0] = c_first;
        gcount[1] = c_last;
      }
    }
    build_tile_list(slot, nslots, tlist, C::TCAP, tcount);
  }
  if (threadIdx.x == 32) {
    mbar_init(q_full, 1);
    mbar_init(q_tmem, 128);
    // gathered tiles: one arrival per producer lane once its copies landed
    for (int i = 0; i < C::KST; ++i) { mbar_init(k_full + i, GAT ? 32 : 1); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < C::VST; ++i) { mbar_init(v_full + i, GAT ? 32 : 1); mbar_init(v_empty + i, 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(s_full + i, 1); mbar_init(p_full + i, 128 * C::NG); }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(fin, 128 * C::NG);
    mbar_init(o_fin, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *tcount;
  const bool any_tile = ntiles > 0;
  if (gat && warp != 0) {
    c_first = gcount[0];
    c_last = gcount[1];
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (!GAT) {
      if (lane == 0 && any_tile) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        mbar_expect_tx(q_full, C::QTILE);
        for (int j = 0; j < C::NQSLAB; ++j) {
          if constexpr (PK)  // packed rows: one row range over all heads
            tma_load_3d(sQ + j * C::QSLAB, &p.tm_q, q_full, j * (C::SWQ / 2), row_base + q0, 0);
          else
            tma_load_3d(sQ + j * C::QSLAB, &p.tm_q, q_full, j * (C::SWQ / 2), q0, bh);
        }
        int n = 0, nk = 0, nv = 0;
        bool ok = true;
        auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
        int kv0;
        bool masked;
        while (ok && it.next(&kv0, &masked)) {
          // (row, head) coordinates of the key/value tile: a dense head, or the
          // page holding the tile in a paged pool (pages hold multiples of 128 keys)
          int ky = kv0, kz = bkv;
          if constexpr (PK) {
            if (p.pk_pages) {
              int page = __ldg(p.pk_pages + (size_t)(bkv / p.Hkv) * p.pk_max_pages + kv0 / p.pk_page_size);
              if (page < 0 || page >= p.pk_num_pages) {
                raise_dev_error(GBATTN_ERR_BLOCKS);  // read page 0 instead; the output is invalid
                page = 0;
              }
              ky = kv0 % p.pk_page_size;
              kz = page * p.Hkv + bkv % p.Hkv;
            }
          }
          const int ks = n % C::KST;
          if (n >= C::KST && !(ok = mbar_wait(k_empty + ks, ((n / C::KST) + 1) & 1, abort_flag))) break;
          if (!(p.test_withhold_k && n == 0)) {
            mbar_expect_tx(k_full + ks, C::QTILE);
            for (int j = 0; j < C::NQSLAB; ++j)
              tma_load_3d(sK + ks * C::QTILE + j * C::QSLAB, &p.tm_k, k_full + ks, j * (C::SWQ / 2), ky, kz);
          }
          ++nk;  // a withheld tile counts too: its drain below gives up after the time limit
          const int vs = n % C::VST;
          if (n >= C::VST && !(ok = mbar_wait(v_empty + vs, ((n / C::VST) + 1) & 1, abort_flag))) break;
          mbar_expect_tx(v_full + vs, C::VTILE);
          for (int j = 0; j < C::NVSLAB; ++j)
            tma_load_3d(sV + vs * C::VTILE + j * C::VSLAB, &p.tm_v, v_full + vs, j * (C::SWV / 2), ky, kz);
          ++nv;
          ++n;
        }
        if (*abort_flag) {
          // let every copy this thread started land before the CTA exits
          mbar_drain(q_full, 0, abort_flag);
          for (int t = (nk > C::KST ? nk - C::KST : 0); t < nk; ++t) mbar_drain(k_full + t % C::KST, (t / C::KST) & 1, abort_flag);
          for (int t = (nv > C::VST ? nv - C::VST : 0); t < nv; ++t) mbar_drain(v_full + t % C::VST, (t / C::VST) & 1, abort_flag);
        }
      }
    } else if (any_tile) {
      // gathered keys: lane 0 waits and issues Q; the warp copies the kept
      // rows of each K and V tile with cp.async (lane l looks up the rows
      // l, l + 32, l + 64 and l + 96 of the tile)
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        mbar_expect_tx(q_full, C::QTILE);
        for (int j = 0; j < C::NQSLAB; ++j) tma_load_3d(sQ + j * C::QSLAB, &p.tm_q, q_full, j * (C::SWQ / 2), q0, bh);
      }
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int kv0;
      bool masked;
      const __nv_bfloat16* kh = p.gk + (size_t)bkv * p.Sk * DQK;
      const __nv_bfloat16* vh = p.gv + (size_t)bkv * p.Sk * DV;
      while (ok && it.next(&kv0, &masked)) {
        int ro[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) ro[e] = __ldg(pos_h + min(kv0 + 32 * e + lane, Skv - 1));
        const int ks = n % C::KST;
        bool w = true;
        if (lane == 0 && n >= C::KST) w = mbar_wait(k_empty + ks, ((n / C::KST) + 1) & 1, abort_flag);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
        // (the empty barrier completes once the tensor cores have read the stage)
        gather_tile_async<DQK, C::SWQ>(sK + ks * C::QTILE, kh, ro, lane);
        cp_async_arrive(k_full + ks);
        const int vs = n % C::VST;
        if (lane == 0 && n >= C::VST) w = mbar_wait(v_empty + vs, ((n / C::VST) + 1) & 1, abort_flag);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
        gather_tile_async<DV, C::SWV>(sV + vs * C::VTILE, vh, ro, lane);
        cp_async_arrive(v_full + vs);
        ++n;
      }
      cp_async_wait_all();  // every copy of this thread lands before the CTA exits
      if (lane == 0 && *abort_flag) mbar_drain(q_full, 0, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && any_tile) {
      const SDesc kd = make_sdesc(smem_u32(sK), 16, 8 * C::SWQ, swz_code(C::SWQ));
      const SDesc vd = make_sdesc(smem_u32(sV), C::VSLAB, 8 * C::SWV, swz_code(C::SWV));
      auto issue_pv = [&](int j) -> bool {
        // the V tile landed long before P_j is written: its wait goes first,
        // so that P_j's arrival is followed directly by the product
        const int sb = j & 1;
        const int vs = j % C::VST;
        if (!mbar_wait(v_full + vs, (j / C::VST) & 1, abort_flag)) return false;
        if (!mbar_wait(p_full + sb, (j >> 1) & 1, abort_flag)) return false;
        if constexpr (GAT) fence_async_smem();  // rows copied with cp.async
        tc_fence_after();
        // B = V tile, MN-major: 16 key rows per step; LBO = slab stride, SBO = 8 rows
        const uint32_t vlo = vd.lo + ((vs * C::VTILE) >> 4);
        const uint32_t pa = tmem + sb * 128;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::T_O, pa + kk * 8, vlo + mnmajor_step(kk, C::SWV), vd.hi, C::IDESC_PV, kk > 0 ? 1u : acc0);
        umma_commit(v_empty + vs);
        umma_commit(o_done);
        return true;
      };
      int n = 0;
      bool ok = mbar_wait(q_tmem, 0, abort_flag);
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int kv0;
      bool masked;
      while (ok && it.next(&kv0, &masked)) {
        const int ks = n % C::KST;
        if (!(ok = mbar_wait(k_full + ks, (n / C::KST) & 1, abort_flag))) break;
        if constexpr (GAT) fence_async_smem();  // rows copied with cp.async
        tc_fence_after();
        const uint32_t d = tmem + (n & 1) * 128;
        const uint32_t klo = kd.lo + ((ks * C::QTILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_ts(d, tmem + C::T_Q + kk * 8, klo + kmajor_step(kk, C::SWQ, C::QSLAB), kd.hi, C::IDESC_S, kk > 0 ? 1u : 0u);
        umma_commit(k_empty + ks);
        umma_commit(s_full + (n & 1));
        if (n >= 1 && !(ok = issue_pv(n - 1))) break;
        ++n;
      }
      if (ok && n >= 1 && issue_pv(n - 1)) umma_commit(o_fin);
      if (*abort_flag) {
        umma_commit(drain);
        mbar_drain(drain, 0, abort_flag);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    constexpr int NG = C::NG, CWF = C::CWF;
    const int sw = warp - 2;       // 0 .. 4 NG - 1
    const int grp = sw >> 2;       // which group of CWF key columns
    const int quarter = warp & 3;  // TMEM lane quarter
    const int row = quarter * 32 + lane;
    // query position of this row (the row itself, or its position within its
    // head when rows are packed), whether it exists, and its output row id
    const int i = PK ? (q0 + row) % p.Sq : q0 + row;
    const bool valid = PK ? q0 + row < p.pk_R : i < p.Sq;
    const bool wact = !PK || q0 + quarter * 32 < p.pk_R;  // some row of this warp exists
    const size_t orow_id = PK ? (size_t)row_base + q0 + row : (size_t)bh * p.Sq + i;
    const int cb = grp * CWF;      // first S column of this thread
    constexpr int DVH = DV / NG;   // O columns of this thread
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    int lo = 0, hi;
    if constexpr (GAT) hi = gathered_row_hi(keep_h, p.mask.nkw, q0 + quarter * 32 + delta);
    else row_interval(p.mask, i, p.Sq, SkM, lo, hi);
    const float* kb = p.mask.key_bias ? p.mask.key_bias + (size_t)bh * p.Sk : nullptr;
    const uint32_t* keep = GAT ? nullptr : keep_h;  // gathered keys are all kept
    if (p.mask.table) keep = i < p.Sq ? table_row(p.mask, bh, p.Sq, i) : nullptr;  // this row's element bits
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0;
    bool ok = true;
    if (any_tile && grp == 0) {
      // copy this thread's Q row from the swizzled smem tile into TMEM
      ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag));
      if (ok) {
        uint32_t qr[DQK / 2];
#pragma unroll
        for (int u = 0; u < DQK / 8; ++u) {
          const int slab = u / (C::SWQ / 16), c16 = u % (C::SWQ / 16);
          const int swz = (row * C::SWQ / 128) & (C::SWQ / 16 - 1);
          const uint4 v = *reinterpret_cast<const uint4*>(sQ + slab * C::QSLAB + row * C::SWQ + ((c16 ^ swz) << 4));
          qr[4 * u] = v.x;
          qr[4 * u + 1] = v.y;
          qr[4 * u + 2] = v.z;
          qr[4 * u + 3] = v.w;
        }
        if constexpr (DQK / 2 >= 32) {
#pragma unroll
          for (int c = 0; c < DQK / 2; c += 32) tmem_st32(tl + C::T_Q + c, qr + c);
        } else {
          tmem_st16(tl + C::T_Q, qr);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(q_tmem);
      }
    }
    auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
    int kv0;
    bool masked;
    auto kt = key_terms<GAT, CWF / 32>(it, kb, pos_h, Skv, cb + lane, p.mask.slope);
    // Every softmax warp walks every tile and meets its lane quarter's other
    // warps at one named barrier per tile (the row-max exchange), which also
    // ORs their failure flags: a warp whose wait gave up goes on to the next
    // exchange without waiting and they all leave the loop there, so no warp
    // is left at a barrier that a departed warp would have to reach.
    while (it.next(&kv0, &masked)) {
      const int sb = n & 1;
      if constexpr (PK) {
        // packed decode: a warp whose 32 rows hold no query row of the group
        // only keeps the barriers in step (S of this tile is computed, so P
        // of the tile two before is consumed and the arrival cannot run ahead)
        if (!wact) {
          if (!ok || !(ok = __all_sync(0xffffffffu, mbar_wait(s_full + sb, (n >> 1) & 1, abort_flag)))) break;
          mbar_arrive(p_full + sb);
          ++n;
          continue;
        }
      }
      // per-key score term (key bias - slope * j) * log2(e) of this warp's CWF
      // columns; each warp keeps its own copy, so only a warp sync is needed
      float* ctw = colterm + (sw * 2 + sb) * CWF;
      kt.emit(kv0, ctw);
      __syncwarp();
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(s_full + sb, (n >> 1) & 1, abort_flag));
      if (!ok) {  // this tile's exchange, reporting the failure: all leave
        bar_red_or(1 + quarter, 32 * NG, true);
        break;
      }
      tc_fence_after();
      float t[CWF];
      if constexpr (CWF == 64) tmem_ld64(tl + sb * 128 + cb, reinterpret_cast<uint32_t*>(t));
      else tmem_ld32(tl + sb * 128 + cb, reinterpret_cast<uint32_t*>(t));
      tmem_wait_ld32(reinterpret_cast<uint32_t*>(t));
      if constexpr (CWF == 64) reg_fence32(reinterpret_cast<uint32_t*>(t) + 32);
      {
        const float4* ct = reinterpret_cast<const float4*>(ctw);
#pragma unroll
        for (int c4 = 0; c4 < CWF / 4; ++c4) {
          const float4 v4 = ct[c4];
          const int c = 4 * c4;
          if constexpr (CAP) {
            const float cv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) t[c + e] = fmaf(p.cap_post, tanh_fast(t[c + e] * p.cap_pre), cv[e]);
          } else {  // two columns per instruction
            fma2(t[c], t[c + 1], t[c], t[c + 1], p.scale_log2, p.scale_log2, v4.x, v4.y);
            fma2(t[c + 2], t[c + 3], t[c + 2], t[c + 3], p.scale_log2, p.scale_log2, v4.z, v4.w);
          }
        }
      }
      if (masked) {
        const int clo = lo - kv0 - cb;
        const int chi = min(hi, Skv - 1) - kv0 - cb;
        if (keep) {
          uint32_t kw[CWF / 32];
#pragma unroll
          for (int w = 0; w < CWF / 32; ++w) {
            const int wi = ((kv0 + cb) >> 5) + w;
            kw[w] = wi < p.mask.nkw ? __ldg(keep + wi) : 0u;
          }
#pragma unroll
          for (int c = 0; c < CWF; ++c) {
            const bool okc = (c >= clo) && (c <= chi) && ((kw[c >> 5] >> (c & 31)) & 1u);
            t[c] = okc ? t[c] : -INFINITY;
          }
        } else {
#pragma unroll
          for (int c = 0; c < CWF; ++c) t[c] = (c >= clo && c <= chi) ? t[c] : -INFINITY;
        }
      }
      // row max: 8 independent chains over this thread's columns (three-input
      // max), then the other column groups'
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if constexpr (CWF == 64) {
          mx[e] = max3(t[e], t[e + 8], t[e + 16]);
          mx[e] = max3(mx[e], t[e + 24], t[e + 32]);
          mx[e] = max3(mx[e], t[e + 40], t[e + 48]);
          mx[e] = fmaxf(mx[e], t[e + 56]);
        } else {
          mx[e] = max3(t[e], t[e + 8], t[e + 16]);
          mx[e] = fmaxf(mx[e], t[e + 24]);
        }
      }
      float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      float* xm = xmax + sb * NG * 128;
      xm[grp * 128 + row] = mt;
      if (bar_red_or(1 + quarter, 32 * NG, false)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int g = 0; g < NG; ++g)
        if (g != grp) mt = fmaxf(mt, xm[g * 128 + row]);
      float m_use = m_run, alpha = 1.f;
      bool resc = false;
      if (mt > m_run + 8.0f) {
        if (m_run != -INFINITY) {
          resc = true;
          alpha = ex2(m_run - mt);
        }
        m_use = mt;
      }
      const float msafe = (m_use == -INFINITY) ? 0.f : m_use;
      float ls[8];  // four chains of column pairs
#pragma unroll
      for (int e = 0; e < 8; ++e) ls[e] = 0.f;
      uint32_t pk[CWF / 2];
#pragma unroll
      for (int c = 0; c < CWF / 2; ++c) {
        float d0, d1;
        sub2(d0, d1, t[2 * c], t[2 * c + 1], msafe, msafe);
        const float a0 = ex2(d0);
        const float a1 = ex2(d1);
        const int q = 2 * (c & 3);
        add2(ls[q], ls[q + 1], ls[q], ls[q + 1], a0, a1);
        pk[c] = pack_bf16(a0, a1);
      }
      const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      l_run = (resc ? l_run * alpha : l_run) + lsum;
      m_run = m_use;
      if (__any_sync(0xffffffffu, resc)) {
        // O must not be in flight: PV of the previous tile has completed.
        // (S of this tile was issued after PV of tile n - 2, so at most one
        // o_done phase is outstanding and the parity wait is exact.)
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n - 1) & 1, abort_flag));
        if (!ok) {  // reported at the next exchange
          ++n;
          continue;
        }
        tc_fence_after();
        if constexpr (DVH >= 32) {
#pragma unroll 1
          for (int c0 = 0; c0 < DVH; c0 += 32) {
            uint32_t orr[32];
            tmem_ld32(tl + C::T_O + grp * DVH + c0, orr);
            tmem_wait_ld32(orr);
#pragma unroll
            for (int c = 0; c < 32; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
            tmem_st32(tl + C::T_O + grp * DVH + c0, orr);
          }
        } else {
          uint32_t orr[16];
          tmem_ld16(tl + C::T_O + grp * DVH, orr);
          tmem_wait_ld16(orr);
#pragma unroll
          for (int c = 0; c < 16; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
          tmem_st16(tl + C::T_O + grp * DVH, orr);
        }
      }
      if constexpr (CWF == 64) tmem_st32(tl + sb * 128 + grp * 32, pk);
      else tmem_st16(tl + sb * 128 + grp * 16, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + sb);
      ++n;
    }
    // ---- epilogue: combine the two halves' row sums, normalise my O half
    if (ok) {
      float l_tot = 0.f;
      if (n > 0) {
        xsum[grp * 128 + row] = l_run;
        mbar_arrive(fin);
        ok = __all_sync(0xffffffffu, mbar_wait(fin, 0, abort_flag));
        if (ok) {
#pragma unroll
          for (int g = 0; g < NG; ++g) l_tot += xsum[g * 128 + row];
        }
      }
      if (ok) {
        const bool live = n > 0 && l_tot > 0.f;
        __nv_bfloat16* orow = p.o + orow_id * DV + grp * DVH;
        // split partials (packed decode with several splits): fp32 O / l and LSE
        const bool part = PK && p.pk_nsplit > 1;
        const size_t prow = (size_t)split * BH * p.Sq + orow_id;
        float* oprow = part ? p.o_part + prow * DV + grp * DVH : nullptr;
        if (!live && valid) {
          if (part) {
#pragma unroll
            for (int c = 0; c < DVH; c += 4) *reinterpret_cast<float4*>(oprow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (grp == 0) p.lse_part[prow] = -INFINITY;
          } else {
#pragma unroll
            for (int c = 0; c < DVH; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
            if (grp == 0 && p.lse) p.lse[orow_id] = -INFINITY;
          }
        }
        if (n > 0 && __all_sync(0xffffffffu, mbar_wait(o_fin, 0, abort_flag))) {
          tc_fence_after();
          const float inv = live ? 1.f / l_tot : 0.f;
          constexpr int CH = DVH >= 32 ? 32 : 16;
#pragma unroll 1
          for (int c0 = 0; c0 < DVH; c0 += CH) {
            uint32_t orr[CH];
            if constexpr (CH == 32) {
              tmem_ld32(tl + C::T_O + grp * DVH + c0, orr);
              tmem_wait_ld32(orr);
            } else {
              tmem_ld16(tl + C::T_O + grp * DVH + c0, orr);
              tmem_wait_ld16(orr);
            }
            if (valid && live && part) {
#pragma unroll
              for (int c = 0; c < CH; c += 4)
                *reinterpret_cast<float4*>(oprow + c0 + c) =
                    make_float4(__uint_as_float(orr[c]) * inv, __uint_as_float(orr[c + 1]) * inv,
                                __uint_as_float(orr[c + 2]) * inv, __uint_as_float(orr[c + 3]) * inv);
            } else if (valid && live) {
              uint32_t pkd[CH / 2];
#pragma unroll
              for (int c = 0; c < CH / 2; ++c)
                pkd[c] = pack_bf16(__uint_as_float(orr[2 * c]) * inv, __uint_as_float(orr[2 * c + 1]) * inv);
#pragma unroll
              for (int c = 0; c < CH / 8; ++c)
                *reinterpret_cast<uint4*>(orow + c0 + 8 * c) =
                    make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]);
            }
          }
          if (grp == 0 && valid && live) {
            const float L_nat = (m_run + __log2f(l_tot)) * kLn2 + p.mask.slope * (float)i;
            if (part) p.lse_part[prow] = L_nat;
            else if (p.lse) p.lse[orow_id] = L_nat;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int DQK, int DV, bool CAP, bool GAT>
static int launch_fwd(const FwdParams& prm, int grid, cudaStream_t st) {
  using C = FwdCfg<DQK, DV>;
  auto kern = fwd_bf16_kernel<DQK, DV, CAP, GAT>;
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(kern, C::SMEM, attr)) return GBATTN_ERR_CUDA;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

template <int DQK, int DV>
static int launch_fwd_cap(const FwdParams& prm, int grid, bool cap, cudaStream_t st) {
  if (prm.gather)
    return cap ? launch_fwd<DQK, DV, true, true>(prm, grid, st) : launch_fwd<DQK, DV, false, true>(prm, grid, st);
  return cap ? launch_fwd<DQK, DV, true, false>(prm, grid, st) : launch_fwd<DQK, DV, false, false>(prm, grid, st);
}

int fwd_bf16_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, const HostMask& m,
                    void* o, float* lse, cudaStream_t st, const FwdTestHook* hook) {
  FwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if (hook) {
    prm.wait_ns = hook->wait_ns;
    prm.test_withhold_k = hook->withhold_first_k_tile;
  }
  const int BH = s.B * s.H;
  const int swq = s.Dqk >= 64 ? 128 : 64, swv = s.Dv >= 64 ? 128 : 64;
  if (!make_tmap_bf16_3d(&prm.tm_q, q, s.Dqk, s.Sq, BH, swq)) return GBATTN_ERR_CUDA;
  const int BHkv = s.B * s.Hkv;
  if (m.gather) {  // rows copied by index, no tensor maps
    prm.gk = static_cast<const __nv_bfloat16*>(k);
    prm.gv = static_cast<const __nv_bfloat16*>(v);
  } else {
    if (!make_tmap_bf16_3d(&prm.tm_k, k, s.Dqk, s.Sk, BHkv, swq)) return GBATTN_ERR_CUDA;
    if (!make_tmap_bf16_3d(&prm.tm_v, v, s.Dv, s.Sk, BHkv, swv)) return GBATTN_ERR_CUDA;
  }
  prm.Hkv = s.Hkv;
  prm.G = s.H / s.Hkv;
  prm.gather = m.gather;
  prm.Skv = m.gather ? m.kept : s.Sk;
  prm.kidx = m.gather ? m.keep_idx : nullptr;
  prm.B = s.B;
  prm.H = s.H;
  prm.Sq = s.Sq;
  prm.Sk = s.Sk;
  prm.nqt = (s.Sq + 127) / 128;
  prm.scale_log2 = scale * kLog2e;
  const bool cap = m.softcap > 0.f;
  if (cap) {
    prm.cap_pre = scale / m.softcap;
    prm.cap_post = m.softcap * kLog2e;
  }
  prm.mask.kind = m.kind;
  prm.mask.window_left = m.window_left;
  prm.mask.block_size = m.block_size;
  prm.mask.prefix_len = m.prefix_len;
  prm.mask.slope = m.slope;
  prm.mask.key_bias = m.key_bias;
  prm.mask.keep = m.kind == GBATTN_MASK_DYNAMIC_TOPK ? m.keep : nullptr;
  prm.mask.table = m.kind == GBATTN_MASK_TABLE ? m.table : nullptr;
  prm.mask.table_per_head = m.table_per_head;
  prm.mask.nkw = (s.Sk + 31) / 32;
  prm.has_lists = m.gather ? 0 : m.has_lists;
  if (prm.has_lists) {
    prm.sub = m.sparse_n / 128;
    prm.nqb = m.nqb;
    prm.nkb = m.nkb;
    prm.sparse_m = m.sparse_m;
    prm.mcnt = m.q_mask_cnt;
    prm.midx = m.q_mask_idx;
    prm.fcnt = m.q_full_cnt;
    prm.fidx = m.q_full_idx;
  }
  prm.o = reinterpret_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  // heads grouped so that a wave's K / V tiles stay in L2
  prm.hgroup = head_group(BH, (long long)(m.gather ? m.kept : s.Sk) * (s.Dqk + s.Dv) * 2 / (s.H / s.Hkv), device_l2_bytes());
  const int grid = prm.nqt * BH;
  if (s.Dqk == 32 && s.Dv == 32) return launch_fwd_cap<32, 32>(prm, grid, cap, st);
  if (s.Dqk == 64 && s.Dv == 64) return launch_fwd_cap<64, 64>(prm, grid, cap, st);
  if (s.Dqk == 128 && s.Dv == 128) return launch_fwd_cap<128, 128>(prm, grid, cap, st);
  if (s.Dqk == 192 && s.Dv == 128) return launch_fwd_cap<192, 128>(prm, grid, cap, st);
  return GBATTN_ERR_UNSUPPORTED;
}

template <int D>
static int launch_packed(const FwdParams& prm, int grid, cudaStream_t st) {
  using C = FwdCfg<D, D>;
  auto kern = fwd_bf16_kernel<D, D, false, false, true>;
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(kern, C::SMEM, attr)) return GBATTN_ERR_CUDA;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int fwd_packed_decode_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                             int num_splits, void* o, float* lse, float* o_part, float* lse_part,
                             const PagedKV* paged, cudaStream_t st) {
  FwdParams prm;
  memset(&prm, 0, sizeof(prm));
  const int sw = s.Dqk >= 64 ? 128 : 64;
  const int BHkv = s.B * s.Hkv;
  // Q as one range of B*H*Sq rows: a group's rows are consecutive
  if (!make_tmap_bf16_3d(&prm.tm_q, q, s.Dqk, s.B * s.H * s.Sq, 1, sw)) return GBATTN_ERR_CUDA;
  if (paged && paged->page_table) {
    // the pool as [num_pages * Hkv heads of page_size rows]
    const int heads = paged->num_pages * s.Hkv;
    if (!make_tmap_bf16_3d(&prm.tm_k, k, s.Dqk, paged->page_size, heads, sw)) return GBATTN_ERR_CUDA;
    if (!make_tmap_bf16_3d(&prm.tm_v, v, s.Dv, paged->page_size, heads, sw)) return GBATTN_ERR_CUDA;
    prm.pk_pages = paged->page_table;
    prm.pk_page_size = paged->page_size;
    prm.pk_max_pages = paged->max_pages;
    prm.pk_num_pages = paged->num_pages;
  } else {
    if (!make_tmap_bf16_3d(&prm.tm_k, k, s.Dqk, s.Sk, BHkv, sw)) return GBATTN_ERR_CUDA;
    if (!make_tmap_bf16_3d(&prm.tm_v, v, s.Dv, s.Sk, BHkv, sw)) return GBATTN_ERR_CUDA;
  }
  if (paged) prm.pk_seqlens = paged->seqlens;
  prm.B = s.B;
  prm.H = s.H;
  prm.Sq = s.Sq;
  prm.Sk = s.Sk;
  prm.Hkv = s.Hkv;
  prm.G = s.H / s.Hkv;
  prm.Skv = s.Sk;
  prm.scale_log2 = scale * kLog2e;
  prm.mask.kind = causal ? GBATTN_MASK_CAUSAL : GBATTN_MASK_NONE;
  prm.mask.window_left = -1;
  prm.mask.nkw = (s.Sk + 31) / 32;
  prm.o = reinterpret_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.pk_R = prm.G * s.Sq;
  prm.pk_nrt = (prm.pk_R + 127) / 128;
  prm.pk_nsplit = num_splits;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  const long long grid = (long long)BHkv * prm.pk_nrt * num_splits;
  if (grid >= (1ll << 31)) return GBATTN_ERR_ARG;
  if (s.Dqk == 64 && s.Dv == 64) return launch_packed<64>(prm, (int)grid, st);
  if (s.Dqk == 128 && s.Dv == 128) return launch_packed<128>(prm, (int)grid, st);
  return GBATTN_ERR_UNSUPPORTED;
}

GB_DEFINE_ERROR_READER(fwd_take_error)

}  // namespace gb
