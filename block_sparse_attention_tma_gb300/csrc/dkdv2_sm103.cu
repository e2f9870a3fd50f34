// dkdv2_sm103.cu - key-parallel dK / dV of the fused attention backward on a
// CTA pair (tcgen05 .cta_group::2): two CTAs on two SMs share each MMA.
//
// Method: "Enable 2CTA for SM100 block-sparse backward" (the 2-CTA backward
// over per-kv-block lists of q-blocks, sub-tiled so that a pair of 128-key
// kernel tiles walks one sparse block's list; QK/V dims 192/128) and
// "Optimize Flash Dynamic Mask Attention Kernel Configurations" (the
// key-parallel "seq-k" backward path).
//
// A cluster of two CTAs owns 256 consecutive keys of one key/value head; CTA
// r holds keys [k0 + 128 r, k0 + 128 r + 128) (K and V tiles), its TMEM
// accumulators and its elementwise warps, exactly as the one-CTA kernel in
// dkdv_sm103.cu does. The even CTA's MMA thread issues every product for
// both CTAs with M = 256 (rows = the pair's keys), so the B operand (the
// query tile's Q or dO, 128 query rows) is split between the two CTAs:
//   S^T  = K Q^T    B = Q rows,   CTA r stages query rows [64 r, 64 r + 64)
//   dP^T = V dO^T   B = dO rows,  likewise
//   dV  += P^T dO   B = dO cols,  CTA r stages dO columns [r Dv/2, (r+1) Dv/2)
//   dK  += dS^T Q   B = Q cols,   CTA r stages Q columns [r Dqk/2, (r+1) Dqk/2)
// Each CTA thus loads as many bytes per query tile as the one-CTA kernel
// (a row half and a column half of Q and of dO) but the MMAs read only half
// of each B operand from its shared memory. No load is multicast.
//
// Synchronisation: the even CTA's barriers gate its MMAs. The odd CTA's
// load barriers are relayed to them by its warp 1 (wait locally, arrive
// remotely); the elementwise warps of both CTAs arrive, one lane per warp,
// on the even CTA's S^T/dP^T-read and P^T/dS^T-written barriers. The MMA
// thread's commits arrive on the barrier at the same offset in both CTAs.
#include "bwd_common.cuh"

namespace gb {

template <int DQK, int DV>
struct Dkdv2Cfg {
  static_assert(DQK >= 128 && DV == 128, "pair kernel shapes");
  static constexpr int SW = 128;                               // K, V, Q-row and dO-row tiles
  static constexpr int KSLAB = 128 * SW, NKSLAB = DQK * 2 / SW, KTILE = 128 * DQK * 2;
  static constexpr int VSLAB = 128 * SW, NVSLAB = DV * 2 / SW, VTILE = 128 * DV * 2;
  static constexpr int QRSLAB = 64 * SW, QRTILE = 64 * DQK * 2;  // 64 query rows, K-major
  static constexpr int GRSLAB = 64 * SW, GRTILE = 64 * DV * 2;
  // column halves, MN-major: Dqk / 2 columns of Q (96 at 192: 64-byte swizzle)
  static constexpr int SWQC = (DQK / 2) % 64 == 0 ? 128 : 64;
  static constexpr int QCSLAB = 128 * SWQC, NQCSLAB = DQK / SWQC, QCTILE = 128 * DQK;
  static constexpr int SWGC = 128;  // Dv / 2 = 64 columns: one slab
  static constexpr int GCSLAB = 128 * SWGC, NGCSLAB = DV / SWGC, GCTILE = 128 * DV;
  static constexpr int QST = 2;
  static constexpr int GST = DQK >= 192 ? 1 : 2;
  static constexpr int NG = 2, CW = 128 / NG;
  static constexpr int THREADS = 64 + 128 * NG;
  static constexpr int NEW = 128 * NG;
  static constexpr int EW_WARPS = 2 * 4 * NG;  // elementwise warps of the pair (one arrival each)
  static constexpr int T_R = 0, T_X = 128, T_DV = 192, T_DK = 192 + DV;
  static_assert(192 + DV + DQK <= 512, "TMEM budget");
  enum { B_KV, B_QF, B_QE = B_QF + QST, B_GF = B_QE + QST, B_GE = B_GF + GST, B_S = B_GE + GST, B_RA, B_P, B_DP, B_RB,
         B_DVD, B_DS, B_DKD, B_DONE, B_DRAIN, B_FIN, NBAR };
  static constexpr int TCAP = 1024;
  static constexpr int SMEM_USED = 1024 + KTILE + VTILE + QST * (QRTILE + QCTILE) + GST * (GRTILE + GCTILE) +
                                   QST * 1024 + 512 * (NG - 1) + 4 * (kMaxGroup + 4) + TCAP * 2 + NBAR * 8 + 32 + 2048;
  static constexpr int SMEM = SMEM_USED;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static constexpr uint32_t ID_ST = idesc_bf16(256, 128, false, false);  // S^T = K Q^T, dP^T = V dO^T
  static constexpr uint32_t ID_DV = idesc_bf16(256, DV, false, true);    // dV += P^T dO
  static constexpr uint32_t ID_DK = idesc_bf16(256, DQK, false, true);   // dK += dS^T Q
};

template <int DQK, int DV, bool CAP, bool DB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Dkdv2Cfg<DQK, DV>::THREADS, 1)
    dkdv2_kernel(const __grid_constant__ BwdParams p) {
  using C = Dkdv2Cfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = sK + C::KTILE;
  uint8_t* sQr = sV + C::VTILE;                 // [QST]
  uint8_t* sQc = sQr + C::QST * C::QRTILE;      // [QST]
  uint8_t* sGr = sQc + C::QST * C::QCTILE;      // [GST]
  uint8_t* sGc = sGr + C::GST * C::GRTILE;      // [GST]
  float* sLD = reinterpret_cast<float*>(sGc + C::GST * C::GCTILE);  // [QST][lse2 128 | delta 128]
  float* sDB = sLD + C::QST * 256;                                    // [NG-1][128]
  int* soff = reinterpret_cast<int*>(sDB + 128 * (C::NG - 1));        // [G + 1]
  uint16_t* tlist = reinterpret_cast<uint16_t*>(soff + kMaxGroup + 4);  // [TCAP]
  uint64_t* bar = reinterpret_cast<uint64_t*>(tlist + C::TCAP);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(tmem_slot + 1), p.wait_ns);
  int* tcount = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int BHkv = p.B * p.Hkv;
  const int pair = blockIdx.x >> 1;
  const int bkv = pair % BHkv;
  const int kp0 = (pair / BHkv) * 256;         // first key of the pair
  const int k0 = kp0 + 128 * (int)rank;        // this CTA's keys
  const int k0o = kp0 + 128 * (int)(rank ^ 1u);  // the other CTA's keys
  const int bq0 = (bkv / p.Hkv) * p.H + (bkv % p.Hkv) * p.G;
  const int nqt = (p.Sq + 127) / 128;
  const int SqP = nqt * 128;
  const int Skv = p.Skv;

  // The pair walks one tile sequence: the query tiles either CTA's keys see.
  // Both key tiles lie in one sparse block (sparse_n is a multiple of 256),
  // so they share its list; each CTA keeps its own element-mask flag (a tile
  // its keys do not see at all is walked as a masked tile: every P is 0).
  TileWalk walk;
  int nslots;
  if (p.G == 1) {
    if (p.has_lists) {
      walk = make_walk(p.kmc, p.kmi, p.kfc, p.kfi, bq0 * p.nkb + kp0 / p.sparse_n, p.nqb, p.sub_q, p.Sq);
      nslots = walk.nslots;
    } else {
      nslots = nqt;
    }
  } else if (p.has_lists) {
    if (warp == 0) {
      int tot = 0;
      for (int g0 = 0; g0 < p.G; g0 += 32) {
        const int g = g0 + lane;
        int ns = 0;
        if (g < p.G)
          ns = make_walk(p.kmc, p.kmi, p.kfc, p.kfi, (bq0 + g) * p.nkb + kp0 / p.sparse_n, p.nqb, p.sub_q, p.Sq).nslots;
        int incl = ns;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (g < p.G) soff[g] = tot + incl - ns;
        tot += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) soff[p.G] = tot;
      __syncwarp();
    }
    nslots = 0;
    if (warp == 0) nslots = soff[p.G];
  } else {
    nslots = p.G * nqt;
  }
  // slot s seen from the key tile starting at kt0
  auto slot_of = [&](int s, int kt0, int* st, bool* masked) -> bool {
    if (p.G == 1)
      return p.has_lists ? walk_slot(walk, s, p.mask, false, kt0, p.Sq, p.Sk, st, masked)
                         : dense_slot(s, p.mask, false, kt0, p.Sq, p.Sk, st, masked);
    int g, q0;
    bool ok;
    if (p.has_lists) {
      int lo = 0, hi = p.G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (soff[mid] <= s) lo = mid;
        else hi = mid - 1;
      }
      g = lo;
      const TileWalk w =
          make_walk(p.kmc, p.kmi, p.kfc, p.kfi, (bq0 + g) * p.nkb + kp0 / p.sparse_n, p.nqb, p.sub_q, p.Sq);
      ok = walk_slot(w, s - soff[g], p.mask, false, kt0, p.Sq, p.Sk, &q0, masked);
    } else {
      g = s / nqt;
      ok = dense_slot(s - g * nqt, p.mask, false, kt0, p.Sq, p.Sk, &q0, masked);
    }
    *st = g * SqP + q0;
    return ok;
  };
  auto slot = [&](int s, int* st, bool* masked) -> bool {
    int st2;
    bool m2;
    if (slot_of(s, k0, st, masked)) return true;
    if (!slot_of(s, k0o, &st2, &m2)) return false;
    *st = st2;
    *masked = true;  // only the other CTA's keys see this tile
    return true;
  };
  if (warp == 0) build_tile_list(slot, nslots, tlist, C::TCAP, tcount);
  if (threadIdx.x == 32) {
    for (int b = 0; b < C::NBAR; ++b) {
      uint32_t cnt = 1;
      if (b == C::B_P || b == C::B_DS || b == C::B_RA || b == C::B_RB) cnt = C::EW_WARPS;
      else if (b == C::B_FIN) cnt = C::NEW - 128;
      else if (lead && (b == C::B_KV || (b >= C::B_QF && b < C::B_QF + C::QST) || (b >= C::B_GF && b < C::B_GF + C::GST)))
        cnt = 2;  // own loads + the odd CTA's relayed arrival
      mbar_init(bar + b, cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *tcount;
  if (p.G > 1 && p.has_lists && warp != 0) nslots = soff[p.G];

  if (warp == 0) {
    // ------------------------------------------------------------ producer (each CTA loads its halves)
    if (lane == 0) {
      int n = 0, nq = 0, ng = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int st;
      bool masked;
      while (ok && it.next(&st, &masked)) {
        const int g = st / SqP, q0 = st - g * SqP;
        const int bq = bq0 + g;
        if (n == 0) {
          mbar_expect_tx(bar + C::B_KV, C::KTILE + C::VTILE);
          for (int j = 0; j < C::NKSLAB; ++j)
            tma_load_3d(sK + j * C::KSLAB, &p.tm_k, bar + C::B_KV, j * (C::SW / 2), k0, bkv);
          for (int j = 0; j < C::NVSLAB; ++j)
            tma_load_3d(sV + j * C::VSLAB, &p.tm_v, bar + C::B_KV, j * (C::SW / 2), k0, bkv);
        }
        const int qs = n % C::QST;
        if (n >= C::QST && !(ok = mbar_wait_cluster(bar + C::B_QE + qs, ((n / C::QST) + 1) & 1, abort_flag))) break;
        mbar_expect_tx(bar + C::B_QF + qs, C::QRTILE + C::QCTILE + 1024);
        for (int j = 0; j < C::NKSLAB; ++j)
          tma_load_3d(sQr + qs * C::QRTILE + j * C::QRSLAB, &p.tm_qr, bar + C::B_QF + qs, j * (C::SW / 2),
                      q0 + 64 * (int)rank, bq);
        for (int j = 0; j < C::NQCSLAB; ++j)
          tma_load_3d(sQc + qs * C::QCTILE + j * C::QCSLAB, &p.tm_qc, bar + C::B_QF + qs,
                      (DQK / 2) * (int)rank + j * (C::SWQC / 2), q0, bq);
        bulk_load(sLD + qs * 256, p.lse2 + (size_t)bq * p.sq_pad + q0, 512, bar + C::B_QF + qs);
        bulk_load(sLD + qs * 256 + 128, p.delta + (size_t)bq * p.sq_pad + q0, 512, bar + C::B_QF + qs);
        ++nq;
        const int gs = n % C::GST;
        if (n >= C::GST && !(ok = mbar_wait_cluster(bar + C::B_GE + gs, ((n / C::GST) + 1) & 1, abort_flag))) break;
        mbar_expect_tx(bar + C::B_GF + gs, C::GRTILE + C::GCTILE);
        for (int j = 0; j < C::NVSLAB; ++j)
          tma_load_3d(sGr + gs * C::GRTILE + j * C::GRSLAB, &p.tm_gr, bar + C::B_GF + gs, j * (C::SW / 2),
                      q0 + 64 * (int)rank, bq);
        for (int j = 0; j < C::NGCSLAB; ++j)
          tma_load_3d(sGc + gs * C::GCTILE + j * C::GCSLAB, &p.tm_do, bar + C::B_GF + gs,
                      (DV / 2) * (int)rank + j * (C::SWGC / 2), q0, bq);
        ++ng;
        ++n;
      }
      if (*abort_flag) {
        // own copies only; on the even CTA a phase may also wait for a relay
        // that never comes, and that drain gives up after the time limit
        if (nq > 0) mbar_drain(bar + C::B_KV, 0, abort_flag);
        for (int t = (nq > C::QST ? nq - C::QST : 0); t < nq; ++t)
          mbar_drain(bar + C::B_QF + t % C::QST, (t / C::QST) & 1, abort_flag);
        for (int t = (ng > C::GST ? ng - C::GST : 0); t < ng; ++t)
          mbar_drain(bar + C::B_GF + t % C::GST, (t / C::GST) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !lead) {
      // ------------------------------------------------------------ relay (odd CTA): its loads -> even CTA's barriers
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int st;
      bool masked;
      while (ok && it.next(&st, &masked)) {
        if (n == 0) {
          if (!(ok = mbar_wait(bar + C::B_KV, 0, abort_flag))) break;
          mbar_arrive_cluster(cluster_addr(bar + C::B_KV, 0));
        }
        const int qs = n % C::QST, gs = n % C::GST;
        if (!(ok = mbar_wait(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag))) break;
        mbar_arrive_cluster(cluster_addr(bar + C::B_QF + qs, 0));
        if (!(ok = mbar_wait(bar + C::B_GF + gs, (n / C::GST) & 1, abort_flag))) break;
        mbar_arrive_cluster(cluster_addr(bar + C::B_GF + gs, 0));
        ++n;
      }
    } else if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer (even CTA, for the pair)
      const SDesc kd = make_sdesc(smem_u32(sK), 16, 8 * C::SW, swz_code(C::SW));     // K, K-major
      const SDesc vd = make_sdesc(smem_u32(sV), 16, 8 * C::SW, swz_code(C::SW));     // V, K-major
      const SDesc qr = make_sdesc(smem_u32(sQr), 16, 8 * C::SW, swz_code(C::SW));    // Q rows, K-major
      const SDesc gr = make_sdesc(smem_u32(sGr), 16, 8 * C::SW, swz_code(C::SW));    // dO rows, K-major
      const SDesc qc = make_sdesc(smem_u32(sQc), C::QCSLAB, 8 * C::SWQC, swz_code(C::SWQC));  // Q cols, MN-major
      const SDesc gc = make_sdesc(smem_u32(sGc), C::GCSLAB, 8 * C::SWGC, swz_code(C::SWGC));  // dO cols, MN-major
      auto issue_dk = [&](int j) {
        const int qs = j % C::QST;
        const uint32_t blo = qc.lo + ((qs * C::QCTILE) >> 4);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma2_ts(tmem + C::T_DK, tmem + C::T_X + kk * 8, blo + mnmajor_step(kk, C::SWQC), qc.hi, C::ID_DK,
                  kk > 0 ? 1u : acc0);
        umma_commit_pair(bar + C::B_DKD);
        umma_commit_pair(bar + C::B_QE + qs);
      };
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int q0;
      bool masked;
      while (ok && it.next(&q0, &masked)) {
        if (n == 0 && !(ok = mbar_wait_cluster(bar + C::B_KV, 0, abort_flag))) break;
        const int qs = n % C::QST;
        if (!(ok = mbar_wait_cluster(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag))) break;
        if (n >= 1 && !(ok = mbar_wait_cluster(bar + C::B_RB, (n - 1) & 1, abort_flag))) break;
        tc_fence_after();
        {
          const uint32_t blo = qr.lo + ((qs * C::QRTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma2_ss(tmem + C::T_R, kd.lo + kmajor_step(kk, C::SW, C::KSLAB), kd.hi,
                    blo + kmajor_step(kk, C::SW, C::QRSLAB), qr.hi, C::ID_ST, kk > 0 ? 1u : 0u);
        }
        umma_commit_pair(bar + C::B_S);
        if (n >= 1) {
          if (!(ok = mbar_wait_cluster(bar + C::B_DS, (n - 1) & 1, abort_flag))) break;
          tc_fence_after();
          issue_dk(n - 1);
        }
        if (!(ok = mbar_wait_cluster(bar + C::B_RA, n & 1, abort_flag))) break;
        const int gs = n % C::GST;
        if (!(ok = mbar_wait_cluster(bar + C::B_GF + gs, (n / C::GST) & 1, abort_flag))) break;
        tc_fence_after();
        {
          const uint32_t blo = gr.lo + ((gs * C::GRTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            mma2_ss(tmem + C::T_R, vd.lo + kmajor_step(kk, C::SW, C::VSLAB), vd.hi,
                    blo + kmajor_step(kk, C::SW, C::GRSLAB), gr.hi, C::ID_ST, kk > 0 ? 1u : 0u);
        }
        umma_commit_pair(bar + C::B_DP);
        if (!(ok = mbar_wait_cluster(bar + C::B_P, n & 1, abort_flag))) break;
        tc_fence_after();
        {
          const uint32_t blo = gc.lo + ((gs * C::GCTILE) >> 4);
          const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma2_ts(tmem + C::T_DV, tmem + C::T_X + kk * 8, blo + mnmajor_step(kk, C::SWGC), gc.hi, C::ID_DV,
                    kk > 0 ? 1u : acc0);
        }
        umma_commit_pair(bar + C::B_DVD);
        umma_commit_pair(bar + C::B_GE + gs);
        ++n;
      }
      if (ok && n >= 1) {
        if ((ok = mbar_wait_cluster(bar + C::B_DS, (n - 1) & 1, abort_flag))) {
          tc_fence_after();
          issue_dk(n - 1);
        }
      }
      umma_commit_pair(bar + C::B_DONE);
      if (*abort_flag) {
        umma_commit_pair(bar + C::B_DRAIN);
        mbar_drain(bar + C::B_DRAIN, 0, abort_flag);
      }
    }
  } else {
    // ------------------------------------------------------------ P / dS warps (own keys)
    constexpr int CW = C::CW;
    const int sw = warp - 2, grp = sw >> 2, cb = grp * CW;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int j = k0 + row;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    // one arrival per warp on the even CTA's barrier
    const uint32_t lb_ra = cluster_addr(bar + C::B_RA, 0), lb_p = cluster_addr(bar + C::B_P, 0);
    const uint32_t lb_rb = cluster_addr(bar + C::B_RB, 0), lb_ds = cluster_addr(bar + C::B_DS, 0);
    auto arrive_lead = [&](uint32_t a) {
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(a);
    };
    int ilo, ihi;
    float kt;
    bool kept;
    auto head_terms = [&](int bq) {
      kept = j < Skv;
      if (kept && p.mask.keep) kept = (__ldg(p.mask.keep + (size_t)bq * p.mask.nkw + (j >> 5)) >> (j & 31)) & 1u;
      const float kb = (j < Skv && p.mask.key_bias) ? __ldg(p.mask.key_bias + (size_t)bq * p.Sk + j) : 0.f;
      kt = (kb - p.mask.slope * (float)j) * kLog2e;
    };
    col_interval(p.mask, j, p.Sq, p.Sk, ilo, ihi);
    head_terms(bq0);
    int g_cur = 0;
    float dbs = 0.f;
    int n = 0;
    bool ok = true;
    auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
    int st;
    bool masked;
    while (ok && it.next(&st, &masked)) {
      int q0 = st;
      if (p.G > 1) {
        const int g = st / SqP;
        q0 = st - g * SqP;
        if (g != g_cur) {
          g_cur = g;
          head_terms(bq0 + g);
        }
      }
      const int qs = n % C::QST;
      ok = mbar_wait_cluster(bar + C::B_S, n & 1, abort_flag);
      if (ok) ok = mbar_wait_cluster(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* sl = sLD + qs * 256;
      const float* sd = sl + 128;
      uint32_t r[CW];
      tmem_ld32(tl + C::T_R + cb, r);
      tmem_ld32(tl + C::T_R + cb + 32, r + 32);
      tmem_wait_ld32(r);
      reg_fence32(r + 32);
      tc_fence_before();
      arrive_lead(lb_ra);
      uint32_t pk[CW / 2], dc[CAP ? CW / 2 : 1];
      const int clo = masked ? (kept ? ilo - q0 : 128) - cb : 0;
      const int chi = masked ? ihi - q0 - cb : CW - 1;
      {
        const float4* sl4 = reinterpret_cast<const float4*>(sl + cb);
        float* pf = reinterpret_cast<float*>(r);
#pragma unroll
        for (int c4 = 0; c4 < CW / 4; ++c4) {
          const float4 l4 = sl4[c4];
          const int c = 4 * c4;
          if constexpr (CAP) {
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            float dd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float th = tanh_fast(__uint_as_float(r[c + e]) * p.cap_pre);
              dd[e] = 1.f - th * th;
              pf[c + e] = ex2(fmaf(p.cap_post, th, kt) - lv[e]);
            }
            dc[2 * c4] = pack_bf16(dd[0], dd[1]);
            dc[2 * c4 + 1] = pack_bf16(dd[2], dd[3]);
          } else {  // two columns per instruction
            float t0, t1, t2, t3;
            fma2(t0, t1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), p.scale_log2, p.scale_log2, kt, kt);
            fma2(t2, t3, __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]), p.scale_log2, p.scale_log2, kt, kt);
            sub2(t0, t1, t0, t1, l4.x, l4.y);
            sub2(t2, t3, t2, t3, l4.z, l4.w);
            pf[c] = ex2(t0);
            pf[c + 1] = ex2(t1);
            pf[c + 2] = ex2(t2);
            pf[c + 3] = ex2(t3);
          }
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < CW; ++c) pf[c] = (c >= clo && c <= chi) ? pf[c] : 0.f;
        }
#pragma unroll
        for (int c = 0; c < CW / 2; ++c) pk[c] = pack_bf16(pf[2 * c], pf[2 * c + 1]);
      }
      if (n >= 1) {
        ok = mbar_wait_cluster(bar + C::B_DKD, (n - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tl + C::T_X + grp * 32, pk);
      tmem_wait_st();
      tc_fence_before();
      arrive_lead(lb_p);
      ok = mbar_wait_cluster(bar + C::B_DP, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(tl + C::T_R + cb, r);
      tmem_ld32(tl + C::T_R + cb + 32, r + 32);
      tmem_wait_ld32(r);
      reg_fence32(r + 32);
      tc_fence_before();
      arrive_lead(lb_rb);
      uint32_t ds[CW / 2];
      {
        const float4* sd4 = reinterpret_cast<const float4*>(sd + cb);
#pragma unroll
        for (int c4 = 0; c4 < CW / 4; ++c4) {
          const float4 d4 = sd4[c4];
          const uint32_t p01 = pk[2 * c4], p23 = pk[2 * c4 + 1];
          float d0 = bf_lo(p01) * (__uint_as_float(r[4 * c4 + 0]) - d4.x);
          float d1 = bf_hi(p01) * (__uint_as_float(r[4 * c4 + 1]) - d4.y);
          float d2 = bf_lo(p23) * (__uint_as_float(r[4 * c4 + 2]) - d4.z);
          float d3 = bf_hi(p23) * (__uint_as_float(r[4 * c4 + 3]) - d4.w);
          if constexpr (DB) dbs += (d0 + d1) + (d2 + d3);
          if constexpr (CAP) {
            d0 *= bf_lo(dc[2 * c4]);
            d1 *= bf_hi(dc[2 * c4]);
            d2 *= bf_lo(dc[2 * c4 + 1]);
            d3 *= bf_hi(dc[2 * c4 + 1]);
          }
          ds[2 * c4] = pack_bf16(d0, d1);
          ds[2 * c4 + 1] = pack_bf16(d2, d3);
        }
      }
      ok = mbar_wait_cluster(bar + C::B_DVD, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32(tl + C::T_X + grp * 32, ds);
      tmem_wait_st();
      tc_fence_before();
      arrive_lead(lb_ds);
      ++n;
    }
    // ---- epilogue: this CTA's dV, dK rows (and key-bias gradient)
    if (ok) {
      const bool wrote = n > 0;
      if (wrote) {
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar + C::B_DONE, 0, abort_flag));
        tc_fence_after();
      }
      const bool jin = j < Skv;
      if constexpr (DB) {
        if (ok && grp >= 1) {
          sDB[(grp - 1) * 128 + row] = dbs;
          mbar_arrive(bar + C::B_FIN);
        } else if (ok && mbar_wait(bar + C::B_FIN, 0, abort_flag) && jin) {
          float t = dbs;
#pragma unroll
          for (int g2 = 0; g2 < C::NG - 1; ++g2) t += sDB[g2 * 128 + row];
          p.dbias[(size_t)bq0 * p.Sk + j] = t;
        }
      }
      if (ok) {
        __nv_bfloat16* dvrow = p.dv + ((size_t)bkv * p.Sk + j) * DV;
        __nv_bfloat16* dkrow = p.dk + ((size_t)bkv * p.Sk + j) * DQK;
#pragma unroll 1
        for (int c0 = grp * 32; c0 < DV + DQK; c0 += 32 * C::NG) {
          const bool isv = c0 < DV;
          uint32_t a[32];
          if (wrote) {
            tmem_ld32(tl + (isv ? C::T_DV + c0 : C::T_DK + c0 - DV), a);
            tmem_wait_ld32(a);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) a[c] = 0u;
          }
          const float sc = isv ? 1.f : p.scale;
          __nv_bfloat16* dst = isv ? dvrow + c0 : dkrow + (c0 - DV);
          if (jin) {
#pragma unroll
            for (int c = 0; c < 32; c += 8)
              *reinterpret_cast<uint4*>(dst + c) =
                  make_uint4(pack_bf16(sc * __uint_as_float(a[c]), sc * __uint_as_float(a[c + 1])),
                             pack_bf16(sc * __uint_as_float(a[c + 2]), sc * __uint_as_float(a[c + 3])),
                             pack_bf16(sc * __uint_as_float(a[c + 4]), sc * __uint_as_float(a[c + 5])),
                             pack_bf16(sc * __uint_as_float(a[c + 6]), sc * __uint_as_float(a[c + 7])));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still touch its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

template <int DQK, int DV, bool CAP, bool DB>
static int launch2_one(const BwdParams& prm, int npairs, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(dkdv2_kernel<DQK, DV, CAP, DB>, Dkdv2Cfg<DQK, DV>::SMEM, attr)) return GBATTN_ERR_CUDA;
  const long long grid = 2ll * npairs * prm.B * prm.Hkv;
  if (grid >= (1ll << 31)) return GBATTN_ERR_ARG;
  dkdv2_kernel<DQK, DV, CAP, DB><<<(unsigned)grid, Dkdv2Cfg<DQK, DV>::THREADS, Dkdv2Cfg<DQK, DV>::SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

template <int DQK, int DV>
static int launch2_cap(const BwdParams& prm, bool cap, bool db, int npairs, cudaStream_t st) {
  if (cap) return db ? launch2_one<DQK, DV, true, true>(prm, npairs, st) : launch2_one<DQK, DV, true, false>(prm, npairs, st);
  return db ? launch2_one<DQK, DV, false, true>(prm, npairs, st) : launch2_one<DQK, DV, false, false>(prm, npairs, st);
}

bool dkdv2_supported(int Dqk, int Dv) { return (Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128); }

int dkdv2_launch(const BwdParams& prm, int Dqk, int Dv, bool cap, bool dbias, int npairs, cudaStream_t st) {
  if (Dqk == 192 && Dv == 128) return launch2_cap<192, 128>(prm, cap, dbias, npairs, st);
  if (Dqk == 128 && Dv == 128) return launch2_cap<128, 128>(prm, cap, dbias, npairs, st);
  return GBATTN_ERR_UNSUPPORTED;
}

GB_DEFINE_ERROR_READER(dkdv2_take_error)

}  // namespace gb
