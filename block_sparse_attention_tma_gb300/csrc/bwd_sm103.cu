// bwd_sm103.cu - fused attention backward on the 5th-generation tensor cores.
//
// Method: "Optimize Flash Dynamic Mask Attention Kernel Configurations"
// (backward with a key-parallel "seq-k" path and a deterministic mode) and
// "Enable 2CTA for SM100 block-sparse backward" (backward walking per-kv-block
// lists of q-blocks, sub-tiled to 128 x 128 kernel tiles; QK/V dims 192/128;
// the rel-bias score_mod passes the gradient through unchanged).
//
// Kernels (the score matrix never reaches memory; dQ needs no atomics, so
// every gradient is bitwise reproducible):
//   bwd_pre      delta_i = sum_d dO_id O_id; lse2_i = LSE_i log2(e) - (row part
//                of the rel bias) in log2 units (+inf for rows with no key or
//                padding rows, so that their P is exactly 0).
//   dkdv         CTA = (b, h, 128-key tile), walking the backward lists over
//                128-row query tiles: S^T = K Q^T and dP^T = V dO^T in TMEM,
//                P^T and dS^T = P^T (dP^T - delta) by the threads owning the
//                key rows, dV += P^T dO and dK += dS^T Q with P^T / dS^T read
//                from TMEM as the A operand.
//   dq           CTA = (b, h, 128-row query tile), walking the forward lists:
//                S = Q K^T, dP = dO V^T, dS = P (dP - delta) -> TMEM,
//                dQ += dS K; dQ is written as bf16 by the same kernel.
// Recomputing S and dP in the dQ kernel costs two extra MMAs per tile pair
// but removes the fp32 dQ accumulator, its atomics and its memory traffic.
//
// Gathered keys (dynamic top-k mask with its kept-key index list): both
// kernels work on compact tiles of kept keys (the dQ kernel copies each tile's
// rows with cp.async, the dK/dV kernel its one K / V tile with TMA row
// gathers); dK / dV
// rows are written back to the keys' original rows and a small kernel zeroes
// the rows of the keys outside the keep set. The key-bias gradient
// (dkey_bias_j = sum_i dS_ij before the softcap factor) is the row sum of
// dS^T that the dK/dV threads already hold, one key row per thread.
#include "bwd_common.cuh"

namespace gb {



// Zeroes dK, dV (and dkey_bias) rows of the keys outside the keep set when
// the kernels gather kept keys only. One warp per (b, h, 32-key word).
__global__ void unkept_zero_kernel(const uint32_t* __restrict__ keep, int nkw, int BH, int Sk, int Dqk, int Dv,
                                   __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                                   float* __restrict__ dbias) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (gw >= (long long)BH * nkw) return;
  const int lane = threadIdx.x & 31;
  const int bh = (int)(gw / nkw), w = (int)(gw % nkw);
  const uint32_t bits = __ldg(keep + gw);
  for (int b = 0; b < 32; ++b) {
    const int j = w * 32 + b;
    if (j >= Sk) break;
    if ((bits >> b) & 1u) continue;
    const size_t r = (size_t)bh * Sk + j;
    for (int c = lane * 8; c < Dqk; c += 256) *reinterpret_cast<uint4*>(dk + r * Dqk + c) = make_uint4(0, 0, 0, 0);
    for (int c = lane * 8; c < Dv; c += 256) *reinterpret_cast<uint4*>(dv + r * Dv + c) = make_uint4(0, 0, 0, 0);
    if (lane == 0 && dbias) dbias[r] = 0.f;
  }
}


// ------------------------------------------------------------------ preprocess
// DV / 8 lanes per row, each loading 16 bytes (8 elements) of O and of dO; a
// warp covers 256 / DV rows, so every load instruction moves 512 contiguous
// bytes of each tensor.
template <int DV>
__global__ void bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ g,
                               const float* __restrict__ lse, int BH, int Sq, int sq_pad, float slope_log2,
                               float* __restrict__ delta, float* __restrict__ lse2) {
  constexpr int LPR = DV / 8, RPW = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const long long gr = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * RPW + lane / LPR;  // padded row
  // every lane stays for the shuffles below; lanes past the last row skip the memory accesses
  const bool in = gr < (long long)BH * sq_pad;
  const int sub = lane % LPR;
  const int bh = in ? (int)(gr / sq_pad) : 0, i = in ? (int)(gr % sq_pad) : 0;
  float d = 0.f, l2 = INFINITY;
  if (in && i < Sq) {
    const size_t row = (size_t)bh * Sq + i;
    const uint4 ov = *reinterpret_cast<const uint4*>(o + row * DV + sub * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(g + row * DV + sub * 8);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
      d = fmaf(a.x, b.x, fmaf(a.y, b.y, d));
    }
    const float L = lse[row];
    l2 = (L == -INFINITY) ? INFINITY : L * kLog2e - slope_log2 * (float)i;
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  if (in && sub == 0) {
    delta[gr] = d;
    lse2[gr] = l2;
  }
}

// ------------------------------------------------------------------ dQ, query-parallel (no atomics)
// CTA = (b, h, 128-row query tile), walking the forward lists (thread = query
// row). Per kv tile n: S_n = Q K_n^T -> [0,128), dP_n = dO V_n^T -> [128,256);
// dS_n = P (dP - delta) -> [448,512) (bf16); dQ += dS_n K_n -> [256,256+Dqk).
// Two threads issue the products (S_n and dP_n from one, dQ_n from the
// other), so the gaps of one issuer are filled by the other's products. The K
// stage of tile n is free once dQ_n is done; the V stage once dP_n is done.
template <int DQK, int DV, bool GAT>
struct DqCfg {
  static constexpr int SWQ = DQK >= 64 ? 128 : 64;
  static constexpr int SWV = DV >= 64 ? 128 : 64;
  static constexpr int QSLAB = 128 * SWQ, NQSLAB = DQK * 2 / SWQ, QTILE = 128 * DQK * 2;
  static constexpr int VSLAB = 128 * SWV, NVSLAB = DV * 2 / SWV, VTILE = 128 * DV * 2;
  // Stages (measured at 8K causal, 16 heads): a third K stage hides the K
  // load behind dQ (Dqk <= 64: shared memory to spare); at Dqk = 128 it costs
  // the second V stage, which the slower cp.async copies of gathered keys
  // cannot spare.
  static constexpr int KST = DQK <= 64 || (DQK == 128 && !GAT) ? 3 : 2;
  static constexpr int VST = DQK >= 192 || (DQK == 128 && !GAT) ? 1 : 2;
  // warp 0 producer, warp 1 S / dP issuer, warps 2..9 elementwise, warp 10 dQ issuer
  static constexpr int THREADS = 352, WDQ = 10;
  static constexpr int T_S = 0, T_DP = 128, T_DQ = 256, T_DS = 448;
  static_assert(T_DQ + DQK <= T_DS, "TMEM budget");
  // B_RS / B_RP: the elementwise warps have copied S / dP out of TMEM;
  // B_DS: dS written to TMEM.
  enum { B_QG, B_KF, B_KE = B_KF + KST, B_VF = B_KE + KST, B_VE = B_VF + VST, B_S = B_VE + VST, B_DP, B_RS, B_RP, B_DS,
         B_DQD, B_DONE, B_DRAIN, B_DRAIN2, NBAR };
  static constexpr int TCAP = 1024;  // visited-tile list entries (uint16)
  static constexpr int SMEM_USED =
      1024 + QTILE + VTILE + KST * QTILE + VST * VTILE + 8 * 2 * 64 * 4 + TCAP * 2 + NBAR * 8 + 32 + 2048;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM
  static constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t ID_DQ = idesc_bf16(128, DQK, false, true);
};

template <int DQK, int DV, bool CAP, bool GAT>
__global__ void __launch_bounds__(DqCfg<DQK, DV, GAT>::THREADS, 1) dq_kernel(const __grid_constant__ BwdParams p) {
  using C = DqCfg<DQK, DV, GAT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sG = sQ + C::QTILE;
  uint8_t* sK = sG + C::VTILE;             // [KST]
  uint8_t* sV = sK + C::KST * C::QTILE;    // [VST]
  float* colterm = reinterpret_cast<float*>(sV + C::VST * C::VTILE);  // [8 warps][2][64]
  uint16_t* tlist = reinterpret_cast<uint16_t*>(colterm + 8 * 128);  // [TCAP]
  uint64_t* bar = reinterpret_cast<uint64_t*>(tlist + C::TCAP);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(tmem_slot + 1), p.wait_ns);
  int* tcount = reinterpret_cast<int*>(tmem_slot + 2);
  int* gcount = reinterpret_cast<int*>(tmem_slot + 4);  // [2] gathered keys seen by the first / last row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int nqt = (p.Sq + 127) / 128;
  int bh, qt;
  grid_tile(blockIdx.x, BH, nqt, p.hgroup, &bh, &qt);
  const int bkv = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;  // key/value head of this query head
  const int q0 = (nqt - 1 - qt) * 128;  // heaviest (last) query tiles first
  constexpr bool gat = GAT;  // gathered keys (compile-time: the list walk keeps its own code)
  const int Skv = p.Skv;
  const int delta = p.Sk - p.Sq;
  const uint32_t* keep_h = p.mask.keep ? p.mask.keep + (size_t)bh * p.mask.nkw : nullptr;
  const int32_t* pos_h = gat ? p.kidx + (size_t)bh * p.Sk : nullptr;

  TileWalk walk;
  int nslots;
  int c_first = 0, c_last = 0;
  if (gat) {
    nslots = (Skv + 127) / 128;
  } else if (p.has_lists) {
    walk = make_walk(p.qmc, p.qmi, p.qfc, p.qfi, bh * p.nqb + q0 / p.sparse_m, p.nkb, p.sub_k, p.Sk);
    nslots = walk.nslots;
  } else {
    nslots = (p.Sk + 127) / 128;
  }
  auto slot = [&](int s, int* kv0, bool* masked) -> bool {
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
    // gathered K / V tiles: one arrival per producer lane once its copies landed
    for (int b = 0; b < C::NBAR; ++b) {
      const bool kv_full = (b >= C::B_KF && b < C::B_KF + C::KST) || (b >= C::B_VF && b < C::B_VF + C::VST);
      mbar_init(bar + b, (b == C::B_DS || b == C::B_RS || b == C::B_RP) ? 256 : (GAT && kv_full) ? 32 : 1);
    }
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
    c_first = gcount[0];
    c_last = gcount[1];
  }

  if (warp == 0) {
    if constexpr (!GAT) {
      if (lane == 0) {
        int n = 0, nk = 0, nv = 0;
        bool ok = true;
        auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
        int kv0;
        bool masked;
        while (ok && it.next(&kv0, &masked)) {
          if (n == 0) {
            mbar_expect_tx(bar + C::B_QG, C::QTILE + C::VTILE);
            for (int j = 0; j < C::NQSLAB; ++j)
              tma_load_3d(sQ + j * C::QSLAB, &p.tm_q, bar + C::B_QG, j * (C::SWQ / 2), q0, bh);
            for (int j = 0; j < C::NVSLAB; ++j)
              tma_load_3d(sG + j * C::VSLAB, &p.tm_do, bar + C::B_QG, j * (C::SWV / 2), q0, bh);
          }
          const int ks = n % C::KST;
          if (n >= C::KST && !(ok = mbar_wait(bar + C::B_KE + ks, ((n / C::KST) + 1) & 1, abort_flag))) break;
          if (!(p.test_withhold && n == 0)) {
            mbar_expect_tx(bar + C::B_KF + ks, C::QTILE);
            for (int j = 0; j < C::NQSLAB; ++j)
              tma_load_3d(sK + ks * C::QTILE + j * C::QSLAB, &p.tm_k, bar + C::B_KF + ks, j * (C::SWQ / 2), kv0,
                          bkv);
          }
          ++nk;  // a withheld tile counts too: its drain below gives up after the time limit
          const int vs = n % C::VST;
          if (n >= C::VST && !(ok = mbar_wait(bar + C::B_VE + vs, ((n / C::VST) + 1) & 1, abort_flag))) break;
          mbar_expect_tx(bar + C::B_VF + vs, C::VTILE);
          for (int j = 0; j < C::NVSLAB; ++j)
            tma_load_3d(sV + vs * C::VTILE + j * C::VSLAB, &p.tm_v, bar + C::B_VF + vs, j * (C::SWV / 2), kv0, bkv);
          ++nv;
          ++n;
        }
        if (*abort_flag) {
          if (nk > 0) mbar_drain(bar + C::B_QG, 0, abort_flag);
          for (int t = (nk > C::KST ? nk - C::KST : 0); t < nk; ++t)
            mbar_drain(bar + C::B_KF + t % C::KST, (t / C::KST) & 1, abort_flag);
          for (int t = (nv > C::VST ? nv - C::VST : 0); t < nv; ++t)
            mbar_drain(bar + C::B_VF + t % C::VST, (t / C::VST) & 1, abort_flag);
        }
      }
    } else {
      // gathered keys: lane 0 waits and issues Q / dO; the warp copies the
      // kept rows of each K and V tile with cp.async (lane l looks up the
      // rows l, l + 32, l + 64 and l + 96 of the tile)
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int kv0;
      bool masked;
      const __nv_bfloat16* kh = p.gk + (size_t)bkv * p.Sk * DQK;
      const __nv_bfloat16* vh = p.gv + (size_t)bkv * p.Sk * DV;
      while (ok && it.next(&kv0, &masked)) {
        if (n == 0 && lane == 0) {
          mbar_expect_tx(bar + C::B_QG, C::QTILE + C::VTILE);
          for (int j = 0; j < C::NQSLAB; ++j)
            tma_load_3d(sQ + j * C::QSLAB, &p.tm_q, bar + C::B_QG, j * (C::SWQ / 2), q0, bh);
          for (int j = 0; j < C::NVSLAB; ++j)
            tma_load_3d(sG + j * C::VSLAB, &p.tm_do, bar + C::B_QG, j * (C::SWV / 2), q0, bh);
        }
        int ro[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) ro[e] = __ldg(pos_h + min(kv0 + 32 * e + lane, Skv - 1));
        // V first: its stage is released by dP of tile n - VST, before the K
        // stage (released by dQ of tile n - KST, issued one tile later). The
        // empty barriers complete once the tensor cores have read the stage.
        const int vs = n % C::VST;
        bool w = true;
        if (lane == 0 && n >= C::VST) w = mbar_wait(bar + C::B_VE + vs, ((n / C::VST) + 1) & 1, abort_flag);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
        gather_tile_async<DV, C::SWV>(sV + vs * C::VTILE, vh, ro, lane);
        cp_async_arrive(bar + C::B_VF + vs);
        const int ks = n % C::KST;
        if (lane == 0 && n >= C::KST) w = mbar_wait(bar + C::B_KE + ks, ((n / C::KST) + 1) & 1, abort_flag);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
        gather_tile_async<DQK, C::SWQ>(sK + ks * C::QTILE, kh, ro, lane);
        cp_async_arrive(bar + C::B_KF + ks);
        ++n;
      }
      cp_async_wait_all();  // every copy of this thread lands before the CTA exits
      if (lane == 0 && *abort_flag && n > 0) mbar_drain(bar + C::B_QG, 0, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S / dP issuer
    // per kv tile n: S_n once S_{n-1} has been copied out, dP_n once dP_{n-1} has
    if (lane == 0) {
      const SDesc qd = make_sdesc(smem_u32(sQ), 16, 8 * C::SWQ, swz_code(C::SWQ));  // Q, K-major
      const SDesc gd = make_sdesc(smem_u32(sG), 16, 8 * C::SWV, swz_code(C::SWV));  // dO, K-major
      const SDesc kd = make_sdesc(smem_u32(sK), 16, 8 * C::SWQ, swz_code(C::SWQ));  // K, K-major
      const SDesc vd = make_sdesc(smem_u32(sV), 16, 8 * C::SWV, swz_code(C::SWV));  // V, K-major
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int kv0;
      bool masked;
      while (ok && it.next(&kv0, &masked)) {
        if (n == 0 && !(ok = mbar_wait(bar + C::B_QG, 0, abort_flag))) break;
        const int ks = n % C::KST, vs = n % C::VST;
        if (!(ok = mbar_wait(bar + C::B_KF + ks, (n / C::KST) & 1, abort_flag))) break;
        if constexpr (GAT) fence_async_smem();  // rows copied with cp.async
        if (n >= 1 && !(ok = mbar_wait(bar + C::B_RS, (n - 1) & 1, abort_flag))) break;  // S_{n-1} read
        tc_fence_after();
        {
          const uint32_t blo = kd.lo + ((ks * C::QTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma_ss(tmem + C::T_S, qd.lo + kmajor_step(kk, C::SWQ, C::QSLAB), qd.hi,
                   blo + kmajor_step(kk, C::SWQ, C::QSLAB), kd.hi, C::ID_S, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar + C::B_S);
        if (!(ok = mbar_wait(bar + C::B_VF + vs, (n / C::VST) & 1, abort_flag))) break;
        if constexpr (GAT) fence_async_smem();  // rows copied with cp.async
        if (n >= 1 && !(ok = mbar_wait(bar + C::B_RP, (n - 1) & 1, abort_flag))) break;  // dP_{n-1} read
        tc_fence_after();
        {
          const uint32_t blo = vd.lo + ((vs * C::VTILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            mma_ss(tmem + C::T_DP, gd.lo + kmajor_step(kk, C::SWV, C::VSLAB), gd.hi,
                   blo + kmajor_step(kk, C::SWV, C::VSLAB), vd.hi, C::ID_S, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar + C::B_DP);
        umma_commit(bar + C::B_VE + vs);
        ++n;
      }
      if (*abort_flag) {
        umma_commit(bar + C::B_DRAIN);
        mbar_drain(bar + C::B_DRAIN, 0, abort_flag);
      }
    }
  } else if (warp == C::WDQ) {
    // ------------------------------------------------------------ dQ issuer
    // per kv tile n: dQ += dS_n K_n once dS_n is in TMEM (S_n, which read the
    // same K stage, completed before the elementwise warps wrote dS_n)
    if (lane == 0) {
      const SDesc km = make_sdesc(smem_u32(sK), C::QSLAB, 8 * C::SWQ, swz_code(C::SWQ));  // K, MN-major
      int n = 0;
      bool ok = true;
      auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
      int kv0;
      bool masked;
      while (ok && it.next(&kv0, &masked)) {
        const int ks = n % C::KST;
        // the K tile landed before S_n was issued: its wait goes first, off
        // the path from the elementwise warps' dS_n to the product
        if (!(ok = mbar_wait(bar + C::B_KF + ks, (n / C::KST) & 1, abort_flag))) break;
        if constexpr (GAT) fence_async_smem();  // rows copied with cp.async
        if (!(ok = mbar_wait(bar + C::B_DS, n & 1, abort_flag))) break;
        tc_fence_after();
        {
          const uint32_t blo = km.lo + ((ks * C::QTILE) >> 4);
          const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_DQ, tmem + C::T_DS + kk * 8, blo + mnmajor_step(kk, C::SWQ), km.hi, C::ID_DQ,
                   kk > 0 ? 1u : acc0);
        }
        umma_commit(bar + C::B_DQD);
        umma_commit(bar + C::B_KE + ks);
        ++n;
      }
      umma_commit(bar + C::B_DONE);
      if (*abort_flag) {
        umma_commit(bar + C::B_DRAIN2);
        mbar_drain(bar + C::B_DRAIN2, 0, abort_flag);
      }
    }
  } else {
    // two warps per TMEM lane quarter; each thread owns one query row and half
    // (64) of the 128 key columns of the tile
    const int sw = warp - 2, grp = sw >> 2, cb = grp * 64;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int i = q0 + row;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    int lo = 0, hi;
    if constexpr (GAT) hi = gathered_row_hi(keep_h, p.mask.nkw, q0 + quarter * 32 + delta);
    else row_interval(p.mask, i, p.Sq, p.Sk, lo, hi);
    const float l2 = p.lse2[(size_t)bh * p.sq_pad + i];
    const float dl = p.delta[(size_t)bh * p.sq_pad + i];
    const float* kb = p.mask.key_bias ? p.mask.key_bias + (size_t)bh * p.Sk : nullptr;
    const uint32_t* keep = gat ? nullptr : keep_h;  // gathered keys are all kept
    if (p.mask.table) keep = i < p.Sq ? table_row(p.mask, bh, p.Sq, i) : nullptr;  // this row's element bits
    int n = 0;
    bool ok = true;
    auto it = tile_seq(slot, tlist, ntiles, C::TCAP, nslots);
    int kv0;
    bool masked;
    // gathered keys: original index -> bias loads run ahead (a dependent pair
    // per tile); otherwise the tile's time hides the one bias load
    auto kt = [&]() {
      if constexpr (GAT) return key_terms<GAT>(it, kb, pos_h, Skv, cb + lane, p.mask.slope);
      else return KeyTermsDirect{kb, Skv, cb + lane, p.mask.slope};
    }();
    while (ok && it.next(&kv0, &masked)) {
      float* ctw = colterm + (sw * 2 + (n & 1)) * 64;
      kt.emit(kv0, ctw);
      __syncwarp();
      uint32_t kw[2] = {0xffffffffu, 0xffffffffu};
      if (keep) {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int wi = ((kv0 + cb) >> 5) + w;
          kw[w] = wi < p.mask.nkw ? __ldg(keep + wi) : 0u;
        }
      }
      const int clo = masked ? lo - kv0 - cb : 0;
      const int chi = masked ? min(hi, Skv - 1) - kv0 - cb : 63;
      ok = mbar_wait(bar + C::B_S, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S: copy out of TMEM (the MMA warp may then reuse it), P in place
      uint32_t rs[64];
      tmem_ld32(tl + C::T_S + cb, rs);
      tmem_ld32(tl + C::T_S + cb + 32, rs + 32);
      tmem_wait_ld32(rs);
      reg_fence32(rs + 32);
      tc_fence_before();
      mbar_arrive(bar + C::B_RS);
      float* pf = reinterpret_cast<float*>(rs);
      float dd[CAP ? 64 : 1];
      {
        const float4* ct = reinterpret_cast<const float4*>(ctw);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 v4 = ct[c4];
          const int c = 4 * c4;
          if constexpr (CAP) {
            const float cv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float th = tanh_fast(__uint_as_float(rs[c + e]) * p.cap_pre);
              dd[c + e] = 1.f - th * th;
              pf[c + e] = ex2(fmaf(p.cap_post, th, cv[e]) - l2);
            }
          } else {  // two columns per instruction
            float t0, t1, t2, t3;
            fma2(t0, t1, __uint_as_float(rs[c]), __uint_as_float(rs[c + 1]), p.scale_log2, p.scale_log2, v4.x, v4.y);
            fma2(t2, t3, __uint_as_float(rs[c + 2]), __uint_as_float(rs[c + 3]), p.scale_log2, p.scale_log2, v4.z,
                 v4.w);
            sub2(t0, t1, t0, t1, l2, l2);
            sub2(t2, t3, t2, t3, l2, l2);
            pf[c] = ex2(t0);
            pf[c + 1] = ex2(t1);
            pf[c + 2] = ex2(t2);
            pf[c + 3] = ex2(t3);
          }
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const bool al = c >= clo && c <= chi && ((kw[c >> 5] >> (c & 31)) & 1u);
            pf[c] = al ? pf[c] : 0.f;
          }
        }
      }
      ok = mbar_wait(bar + C::B_DP, n & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t ds[32];
      {
        uint32_t rp[64];
        tmem_ld32(tl + C::T_DP + cb, rp);
        tmem_ld32(tl + C::T_DP + cb + 32, rp + 32);
        tmem_wait_ld32(rp);
        reg_fence32(rp + 32);
        tc_fence_before();
        mbar_arrive(bar + C::B_RP);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2) {
          // two columns per instruction: (dP - delta), then times P
          float d0, d1;
          sub2(d0, d1, __uint_as_float(rp[2 * c2]), __uint_as_float(rp[2 * c2 + 1]), dl, dl);
          mul2(d0, d1, d0, d1, pf[2 * c2], pf[2 * c2 + 1]);
          if constexpr (CAP) {
            d0 *= dd[2 * c2];
            d1 *= dd[2 * c2 + 1];
          }
          ds[c2] = pack_bf16(d0, d1);
        }
      }
      // the dS columns still feed the dQ MMA of the previous tile
      if (n >= 1) {
        ok = mbar_wait(bar + C::B_DQD, (n - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tl + C::T_DS + grp * 32, ds);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + C::B_DS);
      ++n;
    }
    if (ok) {
      __nv_bfloat16* dst = p.dq + ((size_t)bh * p.Sq + i) * DQK;
      if (n == 0) {
        if (i < p.Sq)
          for (int c = grp * 32; c < DQK; c += 64)
            for (int e = 0; e < 32; e += 8) *reinterpret_cast<uint4*>(dst + c + e) = make_uint4(0, 0, 0, 0);
      } else if (__all_sync(0xffffffffu, mbar_wait(bar + C::B_DONE, 0, abort_flag))) {
        tc_fence_after();
#pragma unroll 1
        for (int c0 = grp * 32; c0 < DQK; c0 += 64) {
          uint32_t a[32];
          tmem_ld32(tl + C::T_DQ + c0, a);
          tmem_wait_ld32(a);
          if (i < p.Sq) {
            const float sc = p.scale;
#pragma unroll
            for (int c = 0; c < 32; c += 8)
              *reinterpret_cast<uint4*>(dst + c0 + c) =
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

// ------------------------------------------------------------------ host
template <int DQK, int DV, bool CAP, bool GAT>
static int launch_dq(const BwdParams& prm, const Shape& s, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(dq_kernel<DQK, DV, CAP, GAT>, DqCfg<DQK, DV, GAT>::SMEM, attr)) return GBATTN_ERR_CUDA;
  dq_kernel<DQK, DV, CAP, GAT>
      <<<((s.Sq + 127) / 128) * s.B * s.H, DqCfg<DQK, DV, GAT>::THREADS, DqCfg<DQK, DV, GAT>::SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

// A second stream of this host thread on the current device, with its fork /
// join events: the dQ grid runs on it beside the dK/dV grid (the two read the
// same inputs and write different outputs), so each grid's CTAs fill the
// other's last wave. Both grids take a whole SM per CTA, so they interleave
// rather than share SMs. Created on first use and kept for the thread's
// lifetime; nullptr (run both on the caller's stream) if creation fails.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
static const SideStream* side_stream() {
  constexpr int kMaxDevices = 64;
  thread_local SideStream ss[kMaxDevices];
  thread_local bool failed[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  SideStream& t = ss[dev];
  if (!t.stream && !failed[dev]) {
    if (cudaStreamCreateWithFlags(&t.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&t.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&t.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      failed[dev] = true;
      t = SideStream{};
    }
  }
  return t.stream ? &t : nullptr;
}

template <int DQK, int DV>
static int launch_dq_cap(const BwdParams& prm, const Shape& s, bool cap, cudaStream_t st) {
  if (prm.gather)
    return cap ? launch_dq<DQK, DV, true, true>(prm, s, st) : launch_dq<DQK, DV, false, true>(prm, s, st);
  return cap ? launch_dq<DQK, DV, true, false>(prm, s, st) : launch_dq<DQK, DV, false, false>(prm, s, st);
}

int bwd_bf16_launch(const Shape& s, const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, float scale, const HostMask& m, void* dq, void* dk, void* dv,
                    float* dkey_bias, void* ws, cudaStream_t st, const BwdTestHook* hook) {
  BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if (hook) {
    prm.wait_ns = hook->wait_ns;
    prm.test_withhold = hook->withhold_first_tiles;
  }
  const int BH = s.B * s.H;
  const int swq = s.Dqk >= 64 ? 128 : 64, swv = s.Dv >= 64 ? 128 : 64;
  if (!make_tmap_bf16_3d(&prm.tm_q, q, s.Dqk, s.Sq, BH, swq)) return GBATTN_ERR_CUDA;
  const int BHkv = s.B * s.Hkv;
  if (m.gather) {
    if (!make_tmap_bf16_rows(&prm.tm_k, k, s.Dqk, (long long)BHkv * s.Sk, swq)) return GBATTN_ERR_CUDA;
    if (!make_tmap_bf16_rows(&prm.tm_v, v, s.Dv, (long long)BHkv * s.Sk, swv)) return GBATTN_ERR_CUDA;
  } else {
    if (!make_tmap_bf16_3d(&prm.tm_k, k, s.Dqk, s.Sk, BHkv, swq)) return GBATTN_ERR_CUDA;
    if (!make_tmap_bf16_3d(&prm.tm_v, v, s.Dv, s.Sk, BHkv, swv)) return GBATTN_ERR_CUDA;
  }
  prm.Hkv = s.Hkv;
  prm.G = s.H / s.Hkv;
  if (!make_tmap_bf16_3d(&prm.tm_do, dout, s.Dv, s.Sq, BH, swv)) return GBATTN_ERR_CUDA;
  prm.gather = m.gather;
  prm.Skv = m.gather ? m.kept : s.Sk;
  prm.kidx = m.gather ? m.keep_idx : nullptr;
  prm.gk = static_cast<const __nv_bfloat16*>(k);
  prm.gv = static_cast<const __nv_bfloat16*>(v);
  prm.dbias = dkey_bias;
  prm.B = s.B;
  prm.H = s.H;
  prm.Sq = s.Sq;
  prm.Sk = s.Sk;
  prm.sq_pad = (int)align_up((size_t)s.Sq, 128);
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  if (m.softcap > 0.f) {
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
    prm.sub_q = m.sparse_m / 128;
    prm.sub_k = m.sparse_n / 128;
    prm.nqb = m.nqb;
    prm.nkb = m.nkb;
    prm.sparse_m = m.sparse_m;
    prm.sparse_n = m.sparse_n;
    prm.qmc = m.q_mask_cnt;
    prm.qmi = m.q_mask_idx;
    prm.qfc = m.q_full_cnt;
    prm.qfi = m.q_full_idx;
    prm.kmc = m.k_mask_cnt;
    prm.kmi = m.k_mask_idx;
    prm.kfc = m.k_full_cnt;
    prm.kfi = m.k_full_idx;
  }
  char* w = static_cast<char*>(ws);
  const size_t vec_bytes = align_up((size_t)BH * prm.sq_pad * sizeof(float), 256);
  float* delta = reinterpret_cast<float*>(w);
  float* lse2 = reinterpret_cast<float*>(w + vec_bytes);
  prm.delta = delta;
  prm.lse2 = lse2;
  // heads grouped so that a wave's streamed tiles stay in L2 (the dQ grid
  // streams K / V, the dK/dV grid Q / dO of every query head of its group)
  prm.hgroup = head_group(BH, (long long)prm.Skv * (s.Dqk + s.Dv) * 2 / prm.G, device_l2_bytes());
  prm.hgroup_kv = head_group(BHkv, (long long)s.Sq * (s.Dqk + s.Dv) * 2 * prm.G, device_l2_bytes());
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);

  {
    const long long rows = (long long)BH * prm.sq_pad;
    const int rpw = 256 / s.Dv;  // rows per warp
    const unsigned blocks = (unsigned)(((rows + rpw - 1) / rpw * 32 + 255) / 256);
    const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(o);
    const __nv_bfloat16* gb_ = static_cast<const __nv_bfloat16*>(dout);
    const float sl2 = m.slope * kLog2e;
    if (s.Dv == 128) bwd_pre_kernel<128><<<blocks, 256, 0, st>>>(ob, gb_, lse, BH, s.Sq, prm.sq_pad, sl2, delta, lse2);
    else if (s.Dv == 64) bwd_pre_kernel<64><<<blocks, 256, 0, st>>>(ob, gb_, lse, BH, s.Sq, prm.sq_pad, sl2, delta, lse2);
    else bwd_pre_kernel<32><<<blocks, 256, 0, st>>>(ob, gb_, lse, BH, s.Sq, prm.sq_pad, sl2, delta, lse2);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  }
  if (m.gather) {
    // rows of the keys outside the keep set: zero gradients
    const long long warps = (long long)BH * prm.mask.nkw;
    unkept_zero_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(
        m.keep, prm.mask.nkw, BH, s.Sk, s.Dqk, s.Dv, prm.dk, prm.dv, dkey_bias);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  }
  const bool cap = m.softcap > 0.f;
  const int nkt = (prm.Skv + 127) / 128;  // key tiles (compact tiles when gathered)
  // dQ on the side stream, forked after the preprocess and joined back
  const SideStream* side = nkt > 0 ? side_stream() : nullptr;
  if (side && (cudaEventRecord(side->fork, st) != cudaSuccess ||
               cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)) {
    cudaGetLastError();
    side = nullptr;
  }
  const cudaStream_t sq = side ? side->stream : st;
  int rc = GBATTN_OK;
  if (nkt > 0) {
    const int key_mode = m.gather ? 1 : (prm.mask.table ? 2 : 0);
    // the CTA-pair dK/dV kernel: closed-form masks (lists whose sparse blocks
    // span both 128-key tiles of a pair), Dqk / Dv = 192 / 128 or 128 / 128
    const bool pair = key_mode == 0 && dkdv2_supported(s.Dqk, s.Dv) && (!prm.has_lists || prm.sparse_n % 256 == 0) &&
                      dkdv_cta_pair_enabled();
    if (pair) {
      const int swqc = (s.Dqk / 2) % 64 == 0 ? 128 : 64;
      if (!make_tmap_bf16_3d_box(&prm.tm_qr, q, s.Dqk, s.Sq, BH, 128, 64) ||
          !make_tmap_bf16_3d_box(&prm.tm_qc, q, s.Dqk, s.Sq, BH, swqc, 128) ||
          !make_tmap_bf16_3d_box(&prm.tm_gr, dout, s.Dv, s.Sq, BH, 128, 64))
        rc = GBATTN_ERR_CUDA;
      else
        rc = dkdv2_launch(prm, s.Dqk, s.Dv, cap, dkey_bias != nullptr, (nkt + 1) / 2, st);
    } else {
      rc = dkdv_launch(prm, s.Dqk, s.Dv, cap, key_mode, dkey_bias != nullptr, nkt * s.B * s.Hkv, st);
    }
  }
  if (rc == GBATTN_OK) {
    if (s.Dqk == 32 && s.Dv == 32) rc = launch_dq_cap<32, 32>(prm, s, cap, sq);
    else if (s.Dqk == 64 && s.Dv == 64) rc = launch_dq_cap<64, 64>(prm, s, cap, sq);
    else if (s.Dqk == 128 && s.Dv == 128) rc = launch_dq_cap<128, 128>(prm, s, cap, sq);
    else if (s.Dqk == 192 && s.Dv == 128) rc = launch_dq_cap<192, 128>(prm, s, cap, sq);
    else rc = GBATTN_ERR_UNSUPPORTED;
  }
  if (side && (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
               cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess))
    return GBATTN_ERR_CUDA;
  return rc;
}

GB_DEFINE_ERROR_READER(bwd_take_error)

}  // namespace gb
