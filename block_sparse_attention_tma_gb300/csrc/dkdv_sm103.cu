// dkdv_sm103.cu - key-parallel dK / dV of the fused attention backward on the
// 5th-generation tensor cores (see bwd_sm103.cu for the whole backward; this
// file holds one kernel family so that it compiles in parallel with the rest).
//
// Method: "Optimize Flash Dynamic Mask Attention Kernel Configurations"
// (backward with a key-parallel "seq-k" path) and "Enable 2CTA for SM100
// block-sparse backward" (per-kv-block lists of q-blocks, QK/V dims 192/128).
#include "bwd_common.cuh"

namespace gb {

// ------------------------------------------------------------------ dK / dV, TMEM-resident (no dQ)
// CTA = (b, h, 128-key tile). Per listed query tile n (thread = key row):
//   S^T_n = K Q_n^T -> R;   P^T_n = exp2(...) -> X (bf16);
//   dP^T_n = V dO_n^T -> R; dV += P^T_n dO_n (A = X);
//   dS^T_n = P^T (dP^T - delta) -> X (bf16);  dK += dS^T_n Q_n (A = X).
// Two threads issue the products: one the score-side S^T_n and dP^T_n
// (writing R), the other the gradient-side dV_n and dK_n (reading X). A
// thread's tcgen05.mma issue keeps pace with the tensor pipe, so every gap
// between its products (a barrier wait, the loop control) would leave the
// pipe idle; with two issuers one thread's gaps are filled by the other's
// products. TMEM: R [0,128), X [128,192), dV [192,192+Dv), dK [192+Dv, +Dqk).
template <int DQK, int DV>
struct DkdvCfg {
  static constexpr int SWQ = DQK >= 64 ? 128 : 64;
  static constexpr int SWV = DV >= 64 ? 128 : 64;
  static constexpr int QSLAB = 128 * SWQ, NQSLAB = DQK * 2 / SWQ, QTILE = 128 * DQK * 2;
  static constexpr int VSLAB = 128 * SWV, NVSLAB = DV * 2 / SWV, VTILE = 128 * DV * 2;
  static constexpr int QST = 2;
  // elementwise warps: NG per TMEM lane quarter, each thread one key row and
  // CW = 128 / NG of the tile's query columns
  static constexpr int NG = 2, CW = 128 / NG;
  // warp 0 producer, warp 1 score-side MMA issuer, warps 2 .. 1 + 4 NG
  // elementwise, warp 2 + 4 NG gradient-side MMA issuer
  static constexpr int THREADS = 64 + 128 * NG + 32;
  static constexpr int WGRAD = 2 + 4 * NG;
  static constexpr int NEW = 128 * NG;  // elementwise threads
  static constexpr int GST = DQK >= 192 ? 1 : 2;
  static constexpr int T_R = 0, T_X = 128, T_DV = 192, T_DK = 192 + DV;
  static_assert(192 + DV + DQK <= 512, "TMEM budget");
  // B_RA / B_RB: the elementwise warps have copied S^T / dP^T out of R (R may
  // be overwritten); B_P / B_DS: P^T / dS^T written to X.
  // B_FIN: the second half's key-bias partial sums are in shared memory.
  // B_GE (dO stage free) completes on two commits: dP^T (score side) and dV
  // (gradient side) both read the stage.
  enum { B_KV, B_QF, B_QE = B_QF + QST, B_GF = B_QE + QST, B_GE = B_GF + GST, B_S = B_GE + GST, B_RA, B_P, B_DP, B_RB,
         B_DVD, B_DS, B_DKD, B_DONE, B_DRAIN, B_DRAIN2, B_FIN, NBAR };
  static constexpr int TCAP = 1024;  // visited-tile list entries (uint16)
  static constexpr int SMEM_USED =
      1024 + QTILE + VTILE + QST * QTILE + GST * VTILE + QST * 1024 + 512 * (NG - 1) + 4 * (kMaxGroup + 4) + TCAP * 2 +
      NBAR * 8 + 32 + 2048;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM
  static constexpr uint32_t ID_ST = idesc_bf16(128, 128, false, false);  // S^T = K Q^T, dP^T = V dO^T
  static constexpr uint32_t ID_DV = idesc_bf16(128, DV, false, true);    // dV += P^T dO
  static constexpr uint32_t ID_DK = idesc_bf16(128, DQK, false, true);   // dK += dS^T Q
};

template <int DQK, int DV, bool CAP, int KM, bool DB>
__global__ void __launch_bounds__(DkdvCfg<DQK, DV>::THREADS, 1) dkdv_kernel(const __grid_constant__ BwdParams p) {
  constexpr bool GAT = KM == 1;  // gathered keys
  constexpr bool TAB = KM == 2;  // element table mask
  using C = DkdvCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = sK + C::QTILE;
  uint8_t* sQ = sV + C::VTILE;                  // [QST]
  uint8_t* sG = sQ + C::QST * C::QTILE;         // [GST]
  float* sLD = reinterpret_cast<float*>(sG + C::GST * C::VTILE);  // [QST][lse2 128 | delta 128]
  float* sDB = sLD + C::QST * 256;                                  // [NG-1][128] key-bias partial sums
  int* soff = reinterpret_cast<int*>(sDB + 128 * (C::NG - 1));      // [G + 1] slot offsets of the query heads
  uint16_t* tlist = reinterpret_cast<uint16_t*>(soff + kMaxGroup + 4);  // [TCAP]
  uint64_t* bar = reinterpret_cast<uint64_t*>(tlist + C::TCAP);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(tmem_slot + 1), p.wait_ns);
  int* tcount = reinterpret_cast<int*>(tmem_slot + 2);
  int* gpos = reinterpret_cast<int*>(tmem_slot + 4);  // [2] first / last key of a gathered tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BHkv = p.B * p.Hkv;
  int bkv, kt;  // key/value head of this CTA and its key tile
  grid_tile(blockIdx.x, BHkv, (p.Skv + 127) / 128, p.hgroup_kv, &bkv, &kt);
  const int k0 = kt * 128;
  // query heads bq0 .. bq0 + G - 1 share this key/value head (GQA); their
  // tiles are walked one head after the other and accumulate into the same
  // dK / dV. A walked tile's start is g * SqP + q0 (g = query head in the group).
  const int bq0 = (bkv / p.Hkv) * p.H + (bkv % p.Hkv) * p.G;
  const int nqt = (p.Sq + 127) / 128;
  const int SqP = nqt * 128;
  constexpr bool gat = GAT;  // gathered keys (compile-time: the list walk keeps its own code)
  const int Skv = p.Skv;
  const int delta = p.Sk - p.Sq;
  const int32_t* pos_h = gat ? p.kidx + (size_t)bq0 * p.Sk : nullptr;

  TileWalk walk;
  int nslots;
  int p_first = 0, p_last = 0;
  if (gat) {
    nslots = nqt;
  } else if (p.G == 1) {
    if (p.has_lists) {
      walk = make_walk(p.kmc, p.kmi, p.kfc, p.kfi, bq0 * p.nkb + k0 / p.sparse_n, p.nqb, p.sub_q, p.Sq);
      nslots = walk.nslots;
    } else {
      nslots = nqt;
    }
  } else if (p.has_lists) {
    // per-head slot counts of the group, prefix-summed into soff by warp 0
    if (warp == 0) {
      int tot = 0;
      for (int g0 = 0; g0 < p.G; g0 += 32) {
        const int g = g0 + lane;
        int ns = 0;
        if (g < p.G) ns = make_walk(p.kmc, p.kmi, p.kfc, p.kfi, (bq0 + g) * p.nkb + k0 / p.sparse_n, p.nqb, p.sub_q,
                                    p.Sq).nslots;
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
    nslots = 0;  // set from soff[G] (after the block-wide barrier for roles other than warp 0)
    if (warp == 0) nslots = soff[p.G];
  } else {
    nslots = p.G * nqt;
  }
  auto slot = [&](int s, int* st, bool* masked) -> bool {
    if (gat) return gathered_slot_cols(s, p_first, p_last, k0 + 128 <= Skv, delta, p.Sq, st, masked);
    if (p.G == 1)
      return p.has_lists ? walk_slot(walk, s, p.mask, false, k0, p.Sq, p.Sk, st, masked)
                         : dense_slot(s, p.mask, false, k0, p.Sq, p.Sk, st, masked);
    int g, q0;
    bool ok;
    if (p.has_lists) {
      int lo = 0, hi = p.G - 1;  // last g with soff[g] <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (soff[mid] <= s) lo = mid;
        else hi = mid - 1;
      }
      g = lo;
      const TileWalk w =
          make_walk(p.kmc, p.kmi, p.kfc, p.kfi, (bq0 + g) * p.nkb + k0 / p.sparse_n, p.nqb, p.sub_q, p.Sq);
      ok = walk_slot(w, s - soff[g], p.mask, false, k0, p.Sq, p.Sk, &q0, masked);
    } else {
      g = s / nqt;
      ok = dense_slot(s - g * nqt, p.mask, false, k0, p.Sq, p.Sk, &q0, masked);
    }
    *st = g * SqP + q0;
    return ok;
  };
  if (warp == 0) {
    if (gat) {
      p_first = __ldg(pos_h + k0);
      p_last = __ldg(pos_h + min(k0 + 127, Skv - 1));
      if (lane == 0) {
        gpos[0] = p_first;
        gpos[1] = p_last;
      }
    }
    build_tile_list(slot, nslots, tlist, C::TCAP, tcount);
  }
  if (threadIdx.x == 32) {
    for (int b = 0; b < C::NBAR; ++b)
      mbar_init(bar + b, (b == C::B_P || b == C::B_DS || b == C::B_RA || b == C::B_RB) ? C::NEW
                         : b == C::B_FIN                                             ? C::NEW - 128
                         : (b >= C::B_GE && b < C::B_GE + C::GST)                   ? 2
                                                                                     : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *tcount;
  if (gat && warp != 0) {
    p_first = gpos[0];
    p_last = gpos[1];
  }
  if (!gat && p.G > 1 && p.has_lists && warp != 0) nslots = soff[p.G];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (!GAT) {
      if (lane == 0) {
        int n = 0, nq = 0, ng = 0;
        bool ok = true;
        auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
        int st;
        bool masked;
        while (ok && it.next(&st, &masked)) {
          const int g = st / SqP, q0 = st - g * SqP;
          const int bq = bq0 + g;  // query head of this tile
          if (n == 0) {
            mbar_expect_tx(bar + C::B_KV, C::QTILE + C::VTILE);
            for (int j = 0; j < C::NQSLAB; ++j)
              tma_load_3d(sK + j * C::QSLAB, &p.tm_k, bar + C::B_KV, j * (C::SWQ / 2), k0, bkv);
            for (int j = 0; j < C::NVSLAB; ++j)
              tma_load_3d(sV + j * C::VSLAB, &p.tm_v, bar + C::B_KV, j * (C::SWV / 2), k0, bkv);
          }
          const int qs = n % C::QST;
          if (n >= C::QST && !(ok = mbar_wait(bar + C::B_QE + qs, ((n / C::QST) + 1) & 1, abort_flag))) break;
          mbar_expect_tx(bar + C::B_QF + qs, C::QTILE + 1024);
          for (int j = 0; j < C::NQSLAB; ++j)
            tma_load_3d(sQ + qs * C::QTILE + j * C::QSLAB, &p.tm_q, bar + C::B_QF + qs, j * (C::SWQ / 2), q0, bq);
          bulk_load(sLD + qs * 256, p.lse2 + (size_t)bq * p.sq_pad + q0, 512, bar + C::B_QF + qs);
          bulk_load(sLD + qs * 256 + 128, p.delta + (size_t)bq * p.sq_pad + q0, 512, bar + C::B_QF + qs);
          ++nq;
          const int gs = n % C::GST;
          if (n >= C::GST && !(ok = mbar_wait(bar + C::B_GE + gs, ((n / C::GST) + 1) & 1, abort_flag))) break;
          if (!(p.test_withhold && n == 0)) {
            mbar_expect_tx(bar + C::B_GF + gs, C::VTILE);
            for (int j = 0; j < C::NVSLAB; ++j)
              tma_load_3d(sG + gs * C::VTILE + j * C::VSLAB, &p.tm_do, bar + C::B_GF + gs, j * (C::SWV / 2), q0, bq);
          }
          ++ng;  // a withheld tile counts too: its drain below gives up after the time limit
          ++n;
        }
        if (*abort_flag) {
          if (nq > 0) mbar_drain(bar + C::B_KV, 0, abort_flag);
          for (int t = (nq > C::QST ? nq - C::QST : 0); t < nq; ++t)
            mbar_drain(bar + C::B_QF + t % C::QST, (t / C::QST) & 1, abort_flag);
          for (int t = (ng > C::GST ? ng - C::GST : 0); t < ng; ++t)
            mbar_drain(bar + C::B_GF + t % C::GST, (t / C::GST) & 1, abort_flag);
        }
      }
    } else {
      // gathered keys: every lane gathers 4 rows of the K and V tiles; lane 0
      // waits and issues the query-side loads
      int n = 0, nq = 0, ng = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int q0;
      bool masked;
      while (ok && it.next(&q0, &masked)) {
        if (n == 0) {
          if (lane == 0) mbar_expect_tx(bar + C::B_KV, C::QTILE + C::VTILE);
          int gr[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) gr[e] = bkv * p.Sk + __ldg(pos_h + min(k0 + 4 * lane + e, Skv - 1));
          __syncwarp();
#pragma unroll
          for (int j = 0; j < C::NQSLAB; ++j)
            tma_gather4(sK + j * C::QSLAB + 4 * lane * C::SWQ, &p.tm_k, bar + C::B_KV, j * (C::SWQ / 2), gr[0], gr[1],
                        gr[2], gr[3]);
#pragma unroll
          for (int j = 0; j < C::NVSLAB; ++j)
            tma_gather4(sV + j * C::VSLAB + 4 * lane * C::SWV, &p.tm_v, bar + C::B_KV, j * (C::SWV / 2), gr[0], gr[1],
                        gr[2], gr[3]);
        }
        if (lane == 0) {
          const int qs = n % C::QST;
          if (n >= C::QST) ok = mbar_wait(bar + C::B_QE + qs, ((n / C::QST) + 1) & 1, abort_flag);
          if (ok) {
            mbar_expect_tx(bar + C::B_QF + qs, C::QTILE + 1024);
            for (int j = 0; j < C::NQSLAB; ++j)
              tma_load_3d(sQ + qs * C::QTILE + j * C::QSLAB, &p.tm_q, bar + C::B_QF + qs, j * (C::SWQ / 2), q0, bq0);
            bulk_load(sLD + qs * 256, p.lse2 + (size_t)bq0 * p.sq_pad + q0, 512, bar + C::B_QF + qs);
            bulk_load(sLD + qs * 256 + 128, p.delta + (size_t)bq0 * p.sq_pad + q0, 512, bar + C::B_QF + qs);
            ++nq;
            const int gs = n % C::GST;
            if (n >= C::GST) ok = mbar_wait(bar + C::B_GE + gs, ((n / C::GST) + 1) & 1, abort_flag);
            if (ok) {
              mbar_expect_tx(bar + C::B_GF + gs, C::VTILE);
              for (int j = 0; j < C::NVSLAB; ++j)
                tma_load_3d(sG + gs * C::VTILE + j * C::VSLAB, &p.tm_do, bar + C::B_GF + gs, j * (C::SWV / 2), q0,
                            bq0);
              ++ng;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++n;
      }
      if (lane == 0 && *abort_flag) {
        if (n > 0) mbar_drain(bar + C::B_KV, 0, abort_flag);
        for (int t = (nq > C::QST ? nq - C::QST : 0); t < nq; ++t)
          mbar_drain(bar + C::B_QF + t % C::QST, (t / C::QST) & 1, abort_flag);
        for (int t = (ng > C::GST ? ng - C::GST : 0); t < ng; ++t)
          mbar_drain(bar + C::B_GF + t % C::GST, (t / C::GST) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score-side MMA issuer
    // per query tile n: S^T_n once dP^T_{n-1} has been copied out of R, then
    // dP^T_n once S^T_n has been
    if (lane == 0) {
      const SDesc kd = make_sdesc(smem_u32(sK), 16, 8 * C::SWQ, swz_code(C::SWQ));  // K, K-major
      const SDesc qd = make_sdesc(smem_u32(sQ), 16, 8 * C::SWQ, swz_code(C::SWQ));  // Q, K-major
      const SDesc vd = make_sdesc(smem_u32(sV), 16, 8 * C::SWV, swz_code(C::SWV));  // V, K-major
      const SDesc gd = make_sdesc(smem_u32(sG), 16, 8 * C::SWV, swz_code(C::SWV));  // dO, K-major
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int q0;
      bool masked;
      while (ok && it.next(&q0, &masked)) {
        if (n == 0 && !(ok = mbar_wait(bar + C::B_KV, 0, abort_flag))) break;
        const int qs = n % C::QST;
        if (!(ok = mbar_wait(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag))) break;
        if (n >= 1 && !(ok = mbar_wait(bar + C::B_RB, (n - 1) & 1, abort_flag))) break;  // dP^T_{n-1} read
        tc_fence_after();
        {
          const uint32_t blo = qd.lo + ((qs * C::QTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma_ss(tmem + C::T_R, kd.lo + kmajor_step(kk, C::SWQ, C::QSLAB), kd.hi,
                   blo + kmajor_step(kk, C::SWQ, C::QSLAB), qd.hi, C::ID_ST, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar + C::B_S);
        // the dO tile lands independently of the elementwise warps (usually
        // before S^T_n has been read): its wait goes first
        const int gs = n % C::GST;
        if (!(ok = mbar_wait(bar + C::B_GF + gs, (n / C::GST) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(bar + C::B_RA, n & 1, abort_flag))) break;  // S^T_n read
        tc_fence_after();
        {
          const uint32_t blo = gd.lo + ((gs * C::VTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            mma_ss(tmem + C::T_R, vd.lo + kmajor_step(kk, C::SWV, C::VSLAB), vd.hi,
                   blo + kmajor_step(kk, C::SWV, C::VSLAB), gd.hi, C::ID_ST, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar + C::B_DP);
        umma_commit(bar + C::B_GE + gs);
        ++n;
      }
      if (*abort_flag) {
        umma_commit(bar + C::B_DRAIN);
        mbar_drain(bar + C::B_DRAIN, 0, abort_flag);
      }
    }
  } else if (warp == C::WGRAD) {
    // ------------------------------------------------------------ gradient-side MMA issuer
    // per query tile n: dV += P^T_n dO_n once P^T_n is in X, then
    // dK += dS^T_n Q_n once dS^T_n is
    if (lane == 0) {
      const SDesc qm = make_sdesc(smem_u32(sQ), C::QSLAB, 8 * C::SWQ, swz_code(C::SWQ));  // Q, MN-major
      const SDesc gm = make_sdesc(smem_u32(sG), C::VSLAB, 8 * C::SWV, swz_code(C::SWV));  // dO, MN-major
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int q0;
      bool masked;
      while (ok && it.next(&q0, &masked)) {
        const uint32_t acc0 = n > 0 ? 1u : 0u;
        // the Q and dO tiles land independently of the elementwise warps
        // (usually before P^T_n is written): their waits go first, off the
        // path from the elementwise warps' arrivals to the products
        const int gs = n % C::GST, qs = n % C::QST;
        if (!(ok = mbar_wait(bar + C::B_GF + gs, (n / C::GST) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(bar + C::B_P, n & 1, abort_flag))) break;  // P^T_n in X
        tc_fence_after();
        {
          const uint32_t blo = gm.lo + ((gs * C::VTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_DV, tmem + C::T_X + kk * 8, blo + mnmajor_step(kk, C::SWV), gm.hi, C::ID_DV,
                   kk > 0 ? 1u : acc0);
        }
        umma_commit(bar + C::B_DVD);
        umma_commit(bar + C::B_GE + gs);
        if (!(ok = mbar_wait(bar + C::B_DS, n & 1, abort_flag))) break;  // dS^T_n in X
        tc_fence_after();
        {
          const uint32_t blo = qm.lo + ((qs * C::QTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_DK, tmem + C::T_X + kk * 8, blo + mnmajor_step(kk, C::SWQ), qm.hi, C::ID_DK,
                   kk > 0 ? 1u : acc0);
        }
        umma_commit(bar + C::B_DKD);
        umma_commit(bar + C::B_QE + qs);
        ++n;
      }
      umma_commit(bar + C::B_DONE);
      if (*abort_flag) {
        umma_commit(bar + C::B_DRAIN2);
        mbar_drain(bar + C::B_DRAIN2, 0, abort_flag);
      }
    }
  } else {
    // ------------------------------------------------------------ P / dS warps
    // NG warps per TMEM lane quarter; each thread owns one key row and CW of
    // the 128 query columns of the tile
    constexpr int CW = C::CW;
    const int sw = warp - 2, grp = sw >> 2, cb = grp * CW;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row
    const int j = k0 + row;  // key (compact index when gathered)
    // original key index (recomputed where needed, to keep registers free)
    auto orig = [&]() -> int { return gat ? (j < Skv ? __ldg(pos_h + j) : 0) : j; };
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    int ilo, ihi;
    float kt;  // per-key score term, log2 units
    bool kept;
    // the keep bit and the key-bias term belong to the query head (bq)
    auto head_terms = [&](int bq) {
      const int jo = orig();
      kept = j < Skv;
      if (kept && p.mask.keep && !gat)
        kept = (__ldg(p.mask.keep + (size_t)bq * p.mask.nkw + (j >> 5)) >> (j & 31)) & 1u;
      const float kb = (j < Skv && p.mask.key_bias) ? __ldg(p.mask.key_bias + (size_t)bq * p.Sk + jo) : 0.f;
      kt = (kb - p.mask.slope * (float)jo) * kLog2e;
    };
    if (gat) {
      ilo = max(0, orig() - delta);
      ihi = p.Sq - 1;
    } else {
      col_interval(p.mask, j, p.Sq, p.Sk, ilo, ihi);
    }
    head_terms(bq0);
    int g_cur = 0;
    float dbs = 0.f;  // key-bias gradient: this half's sum of dS^T (before the softcap factor)
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
      // lse2 / delta landed with Q, before S^T_n was issued: that wait goes
      // first, off the path from S^T_n's completion to the copy-out
      ok = mbar_wait(bar + C::B_QF + qs, (n / C::QST) & 1, abort_flag);
      if (ok) ok = mbar_wait(bar + C::B_S, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* sl = sLD + qs * 256;
      const float* sd = sl + 128;
      // copy S^T out of R, then let the MMA warp reuse R for dP^T
      uint32_t r[CW];
      tmem_ld32(tl + C::T_R + cb, r);
      if constexpr (CW == 64) tmem_ld32(tl + C::T_R + cb + 32, r + 32);
      tmem_wait_ld32(r);
      if constexpr (CW == 64) reg_fence32(r + 32);
      tc_fence_before();
      mbar_arrive(bar + C::B_RA);
      // P^T = exp2(S^T * scale * log2e + key term - lse2[q])
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
          if constexpr (TAB) {
            // element table: lane l fetches the word of query rows cb + l (and
            // cb + 32 + l) that holds this warp's 32 keys (k0 is a multiple of
            // 128, so the word is warp-uniform and bit l is this thread's key)
            const int jw = j >> 5;
            const int bq = bq0 + g_cur;
#pragma unroll
            for (int h = 0; h < CW / 32; ++h) {
              const int rq = q0 + cb + 32 * h + lane;
              const uint32_t w = (rq < p.Sq && jw < p.mask.nkw) ? __ldg(table_row(p.mask, bq, p.Sq, rq) + jw) : 0u;
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((__shfl_sync(0xffffffffu, w, c) >> lane) & 1u)) pf[32 * h + c] = 0.f;
            }
          }
        }
#pragma unroll
        for (int c = 0; c < CW / 2; ++c) pk[c] = pack_bf16_prob(pf[2 * c], pf[2 * c + 1]);
      }
      // X still holds dS^T of the previous tile until its dK MMA completes
      if (n >= 1) {
        ok = mbar_wait(bar + C::B_DKD, (n - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if constexpr (CW == 64) tmem_st32(tl + C::T_X + grp * 32, pk);
      else tmem_st16(tl + C::T_X + grp * 16, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + C::B_P);
      // dP^T: copy out of R (then R is free for S^T of the next tile), dS^T = P^T (dP^T - delta[q])
      ok = mbar_wait(bar + C::B_DP, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(tl + C::T_R + cb, r);
      if constexpr (CW == 64) tmem_ld32(tl + C::T_R + cb + 32, r + 32);
      tmem_wait_ld32(r);
      if constexpr (CW == 64) reg_fence32(r + 32);
      tc_fence_before();
      mbar_arrive(bar + C::B_RB);
      uint32_t ds[CW / 2];
      {
        const float4* sd4 = reinterpret_cast<const float4*>(sd + cb);
#pragma unroll
        for (int c4 = 0; c4 < CW / 4; ++c4) {
          const float4 d4 = sd4[c4];
          const uint32_t p01 = pk[2 * c4], p23 = pk[2 * c4 + 1];
          // two columns per instruction: (dP^T - delta), then times P^T
          float d0, d1, d2, d3;
          sub2(d0, d1, __uint_as_float(r[4 * c4 + 0]), __uint_as_float(r[4 * c4 + 1]), d4.x, d4.y);
          sub2(d2, d3, __uint_as_float(r[4 * c4 + 2]), __uint_as_float(r[4 * c4 + 3]), d4.z, d4.w);
          mul2(d0, d1, d0, d1, bf_lo(p01), bf_hi(p01));
          mul2(d2, d3, d2, d3, bf_lo(p23), bf_hi(p23));
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
      // X holds P^T until the dV MMA completes
      ok = mbar_wait(bar + C::B_DVD, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if constexpr (CW == 64) tmem_st32(tl + C::T_X + grp * 32, ds);
      else tmem_st16(tl + C::T_X + grp * 16, ds);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + C::B_DS);
      ++n;
    }
    // ---- epilogue: dV, dK rows of this thread's key (32-column chunks split
    // between the NG warps of a lane quarter)
    if (ok) {
      const bool wrote = n > 0;
      if (wrote) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar + C::B_DONE, 0, abort_flag));
        tc_fence_after();
      }
      const bool jin = j < Skv;
      const int jo = orig();
      if constexpr (DB) {
        // key-bias gradient of this key: the NG column groups' sums
        if (ok && grp >= 1) {
          sDB[(grp - 1) * 128 + row] = dbs;
          mbar_arrive(bar + C::B_FIN);
        } else if (ok && mbar_wait(bar + C::B_FIN, 0, abort_flag) && jin) {
          float t = dbs;
#pragma unroll
          for (int g2 = 0; g2 < C::NG - 1; ++g2) t += sDB[g2 * 128 + row];
          p.dbias[(size_t)bq0 * p.Sk + jo] = t;
        }
      }
      if (ok) {
        __nv_bfloat16* dvrow = p.dv + ((size_t)bkv * p.Sk + jo) * DV;
        __nv_bfloat16* dkrow = p.dk + ((size_t)bkv * p.Sk + jo) * DQK;
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
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int DQK, int DV, bool CAP, int KM, bool DB>
static int launch_one(const BwdParams& prm, int grid, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(dkdv_kernel<DQK, DV, CAP, KM, DB>, DkdvCfg<DQK, DV>::SMEM, attr)) return GBATTN_ERR_CUDA;
  dkdv_kernel<DQK, DV, CAP, KM, DB><<<grid, DkdvCfg<DQK, DV>::THREADS, DkdvCfg<DQK, DV>::SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

template <int DQK, int DV, bool CAP, int KM>
static int launch_db(const BwdParams& prm, bool db, int grid, cudaStream_t st) {
  return db ? launch_one<DQK, DV, CAP, KM, true>(prm, grid, st) : launch_one<DQK, DV, CAP, KM, false>(prm, grid, st);
}

template <int DQK, int DV, bool CAP>
static int launch_km(const BwdParams& prm, int km, bool db, int grid, cudaStream_t st) {
  if (km == 1) return launch_db<DQK, DV, CAP, 1>(prm, db, grid, st);
  if (km == 2) return launch_db<DQK, DV, CAP, 2>(prm, db, grid, st);
  return launch_db<DQK, DV, CAP, 0>(prm, db, grid, st);
}

template <int DQK, int DV>
static int launch_cap(const BwdParams& prm, bool cap, int km, bool db, int grid, cudaStream_t st) {
  return cap ? launch_km<DQK, DV, true>(prm, km, db, grid, st) : launch_km<DQK, DV, false>(prm, km, db, grid, st);
}

int dkdv_launch(const BwdParams& prm, int Dqk, int Dv, bool cap, int key_mode, bool dbias, int grid, cudaStream_t st) {
  if (Dqk == 32 && Dv == 32) return launch_cap<32, 32>(prm, cap, key_mode, dbias, grid, st);
  if (Dqk == 64 && Dv == 64) return launch_cap<64, 64>(prm, cap, key_mode, dbias, grid, st);
  if (Dqk == 128 && Dv == 128) return launch_cap<128, 128>(prm, cap, key_mode, dbias, grid, st);
  if (Dqk == 192 && Dv == 128) return launch_cap<192, 128>(prm, cap, key_mode, dbias, grid, st);
  return GBATTN_ERR_UNSUPPORTED;
}

GB_DEFINE_ERROR_READER(dkdv_take_error)

}  // namespace gb
