// bwd_common.cuh - parameter block and small helpers shared by the backward
// kernels (dkdv_sm103.cu: key-parallel dK/dV; bwd_sm103.cu: preprocess,
// query-parallel dQ and the host launcher).
#pragma once

#include "kernels.h"
#include "mask.cuh"

namespace gb {

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  // CTA-pair dK/dV kernel: the halves of the Q and dO tiles each CTA stages
  // (query rows [64r, 64r + 64): 64-row boxes; head-dim columns: tm_qc)
  CUtensorMap tm_qr, tm_qc, tm_gr;
  int B, H, Sq, Sk, sq_pad;
  int Hkv, G;          // key/value heads and query heads per key/value head (GQA)
  float scale_log2, cap_pre, cap_post, scale;
  MaskParams mask;
  int has_lists, sub_q, sub_k, nqb, nkb, sparse_m, sparse_n;
  const int32_t *qmc, *qmi, *qfc, *qfi;
  const int32_t *kmc, *kmi, *kfc, *kfi;
  const float* lse2;   // [BH][sq_pad]
  const float* delta;  // [BH][sq_pad]
  __nv_bfloat16 *dq, *dk, *dv;
  float* dbias;        // [BH][Sk] key-bias gradient, or nullptr
  int gather;          // gathered keys: tm_k / tm_v are 2-D row-gather maps (dK/dV
                       // kernel); the dQ kernel copies rows of gk / gv by index
  int Skv;             // key extent the kernels stream (Sk, or the kept-key count)
  const int32_t* kidx; // [BH][Sk] kept key indices (gathered keys)
  const __nv_bfloat16 *gk, *gv;  // K [B*H*Sk, Dqk], V [B*H*Sk, Dv] (gathered keys)
  unsigned long long wait_ns;     // time limit of every wait (0 = kWaitLimitNs)
  int test_withhold;              // test hook: the first dO tile (dK/dV) / K tile (dQ) is never loaded
  int hgroup;                     // dQ grid order: query heads per group (head_group), 0 = none
  int hgroup_kv;                  // dK/dV grid order: key/value heads per group
};

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Launches the dK/dV kernel for one head-dim pair, softcap flag, key mode
// (0: list walk, 1: gathered keys, 2: element table) and key-bias flag.
int dkdv_launch(const BwdParams& prm, int Dqk, int Dv, bool cap, int key_mode, bool dbias, int grid, cudaStream_t st);
// The CTA-pair (cta_group::2) dK/dV kernel: a cluster of two CTAs per 256
// keys. Closed-form masks with or without lists (sparse_n a multiple of 256),
// Dqk / Dv = 192 / 128 or 128 / 128. npairs = pairs of 128-key tiles per
// key/value head. Returns GBATTN_ERR_UNSUPPORTED for other shapes.
int dkdv2_launch(const BwdParams& prm, int Dqk, int Dv, bool cap, bool dbias, int npairs, cudaStream_t st);
bool dkdv2_supported(int Dqk, int Dv);

}  // namespace gb
