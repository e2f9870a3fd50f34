// simt_fp32.cu - exact-fp32 attention forward and backward on CUDA cores.
//
// The fp32 workload of "POPCORNBENCH Kimi-K2.6 l1_p97" asks for fp32 SDPA
// within atol = rtol = 1e-4, which TF32 tensor-core products cannot meet;
// this path therefore multiplies in fp32 FMA. It walks the same block-sparse
// lists and 128-wide kernel tiles as the tensor-core path (same masks,
// softcap and biases), streaming 32-key (or 32-query) chunks through shared
// memory. The backward is deterministic by construction: dQ is computed by a
// query-parallel kernel and dK/dV by a key-parallel kernel, with no atomics.
#include "kernels.h"
#include "mask.cuh"

namespace gb {

constexpr int kSimtThreads = 256;  // 8 warps, 16 rows (or keys) each
constexpr int kChunk = 32;

struct SimtParams {
  int B, H, Sq, Sk, Dqk, Dv;
  int Hkv, G;  // key/value heads, query heads per key/value head (GQA)
  float scale;
  float softcap;
  MaskParams mask;
  int has_lists, sub_q, sub_k, nqb, nkb, sparse_m, sparse_n;
  const int32_t *qmc, *qmi, *qfc, *qfi;  // forward lists (per q-block)
  const int32_t *kmc, *kmi, *kfc, *kfi;  // backward lists (per k-block)
  const float *q, *k, *v, *o, *dout, *lse;
  float *out, *lse_out, *dq, *dk, *dv, *delta;
  float* dbias;  // [B*H, Sk] key-bias gradient, or nullptr
};

// Score of (i, j) from a raw dot product, in natural-log units, and the
// softcap derivative factor d(score)/d(raw scaled dot) (1 without softcap).
__device__ __forceinline__ float simt_score(const SimtParams& p, float dot, int i, int j, const float* kb,
                                            float* dcap) {
  float r = dot * p.scale;
  float s = r;
  *dcap = 1.f;
  if (p.softcap > 0.f) {
    const float t = tanhf(r / p.softcap);
    s = p.softcap * t;
    *dcap = 1.f - t * t;
  }
  if (p.mask.slope != 0.f) s += p.mask.slope * (float)(i - j);
  if (kb) s += kb[j];
  return s;
}

__device__ __forceinline__ bool simt_allowed(const SimtParams& p, int bh, int i, int j, int lo, int hi,
                                             const uint32_t* keep) {
  if (j < lo || j > hi || j >= p.Sk || i >= p.Sq) return false;
  if (keep) return (__ldg(keep + (j >> 5)) >> (j & 31)) & 1u;
  if (p.mask.table) return (__ldg(table_row(p.mask, bh, p.Sq, i) + (j >> 5)) >> (j & 31)) & 1u;
  return true;
}

// ------------------------------------------------------------------ forward
// CTA = (b, h, 128-row query tile); warp w owns rows 16 w .. 16 w + 15.
__global__ void __launch_bounds__(kSimtThreads) simt_fwd_kernel(const SimtParams p) {
  extern __shared__ float sm[];
  const int DQ = p.Dqk, DV = p.Dv;
  float* sQ = sm;                        // [128][DQ]
  float* sK = sQ + 128 * DQ;             // [32][DQ + 1]
  float* sV = sK + kChunk * (DQ + 1);    // [32][DV]
  const int bh = blockIdx.x % (p.B * p.H);
  const int q0 = (blockIdx.x / (p.B * p.H)) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* Q = p.q + (size_t)bh * p.Sq * DQ;
  const int bkv = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;  // key/value head
  const float* K = p.k + (size_t)bkv * p.Sk * DQ;
  const float* V = p.v + (size_t)bkv * p.Sk * DV;
  const float* kb = p.mask.key_bias ? p.mask.key_bias + (size_t)bh * p.Sk : nullptr;
  const uint32_t* keep = p.mask.keep ? p.mask.keep + (size_t)bh * p.mask.nkw : nullptr;

  for (int e = threadIdx.x; e < 128 * DQ; e += blockDim.x) {
    const int r = e / DQ, d = e % DQ;
    sQ[e] = (q0 + r < p.Sq) ? Q[(size_t)(q0 + r) * DQ + d] : 0.f;
  }
  float m[16], l[16], acc[16][4];
  int lo[16], hi[16];
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[rr][t] = 0.f;
    row_interval(p.mask, q0 + warp * 16 + rr, p.Sq, p.Sk, lo[rr], hi[rr]);
  }
  TileWalk walk;
  int nslots;
  if (p.has_lists) {
    walk = make_walk(p.qmc, p.qmi, p.qfc, p.qfi, bh * p.nqb + q0 / p.sparse_m, p.nkb, p.sub_k, p.Sk);
    nslots = walk.nslots;
  } else {
    nslots = (p.Sk + 127) / 128;
  }
  for (int s = 0; s < nslots; ++s) {
    int kv0;
    bool masked;
    const bool ok = p.has_lists ? walk_slot(walk, s, p.mask, true, q0, p.Sq, p.Sk, &kv0, &masked)
                                : dense_slot(s, p.mask, true, q0, p.Sq, p.Sk, &kv0, &masked);
    if (!ok) continue;
    for (int c0 = kv0; c0 < kv0 + 128 && c0 < p.Sk; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * DQ; e += blockDim.x) {
        const int r = e / DQ, d = e % DQ;
        sK[r * (DQ + 1) + d] = (c0 + r < p.Sk) ? K[(size_t)(c0 + r) * DQ + d] : 0.f;
      }
      for (int e = threadIdx.x; e < kChunk * DV; e += blockDim.x) {
        const int r = e / DV, d = e % DV;
        sV[e] = (c0 + r < p.Sk) ? V[(size_t)(c0 + r) * DV + d] : 0.f;
      }
      __syncthreads();
      const int j = c0 + lane;
#pragma unroll 1
      for (int rr = 0; rr < 16; ++rr) {
        const int row = warp * 16 + rr, i = q0 + row;
        float dot = 0.f;
        for (int d = 0; d < DQ; ++d) dot = fmaf(sQ[row * DQ + d], sK[lane * (DQ + 1) + d], dot);
        float dcap;
        float sc = simt_score(p, dot, i, j, kb, &dcap);
        if (!simt_allowed(p, bh, i, j, lo[rr], hi[rr], keep)) sc = -INFINITY;
        float mx = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float mn = fmaxf(m[rr], mx);
        const float msafe = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = (m[rr] == -INFINITY) ? 0.f : expf(m[rr] - msafe);
        const float pj = (sc == -INFINITY) ? 0.f : expf(sc - msafe);
        float ps = pj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l[rr] = l[rr] * alpha + ps;
        m[rr] = mn;
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[rr][t] *= alpha;
        for (int jj = 0; jj < kChunk; ++jj) {
          const float pb = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int d = lane + 32 * t;
            if (d < DV) acc[rr][t] = fmaf(pb, sV[jj * DV + d], acc[rr][t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int i = q0 + warp * 16 + rr;
    if (i >= p.Sq) continue;
    const bool live = l[rr] > 0.f;
    const float inv = live ? 1.f / l[rr] : 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int d = lane + 32 * t;
      if (d < DV) p.out[((size_t)bh * p.Sq + i) * DV + d] = acc[rr][t] * inv;
    }
    if (lane == 0 && p.lse_out) p.lse_out[(size_t)bh * p.Sq + i] = live ? m[rr] + logf(l[rr]) : -INFINITY;
  }
}

// ------------------------------------------------------------------ backward
// delta_i = sum_d dO_id O_id
__global__ void simt_delta_kernel(const SimtParams p) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)p.B * p.H * p.Sq) return;
  const float* o = p.o + gw * p.Dv;
  const float* g = p.dout + gw * p.Dv;
  float s = 0.f;
  for (int d = lane; d < p.Dv; d += 32) s = fmaf(o[d], g[d], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) p.delta[gw] = s;
}

// dQ: CTA = (b, h, 128-row query tile), same walk as the forward.
__global__ void __launch_bounds__(kSimtThreads) simt_dq_kernel(const SimtParams p) {
  extern __shared__ float sm[];
  const int DQ = p.Dqk, DV = p.Dv;
  float* sQ = sm;                         // [128][DQ]
  float* sG = sQ + 128 * DQ;              // [128][DV] dO
  float* sK = sG + 128 * DV;              // [32][DQ + 1]
  float* sV = sK + kChunk * (DQ + 1);     // [32][DV + 1]
  const int bh = blockIdx.x % (p.B * p.H);
  const int q0 = (blockIdx.x / (p.B * p.H)) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bkv = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;  // key/value head
  const float* K = p.k + (size_t)bkv * p.Sk * DQ;
  const float* V = p.v + (size_t)bkv * p.Sk * DV;
  const float* kb = p.mask.key_bias ? p.mask.key_bias + (size_t)bh * p.Sk : nullptr;
  const uint32_t* keep = p.mask.keep ? p.mask.keep + (size_t)bh * p.mask.nkw : nullptr;
  for (int e = threadIdx.x; e < 128 * DQ; e += blockDim.x) {
    const int r = e / DQ, d = e % DQ;
    sQ[e] = (q0 + r < p.Sq) ? p.q[((size_t)bh * p.Sq + q0 + r) * DQ + d] : 0.f;
  }
  for (int e = threadIdx.x; e < 128 * DV; e += blockDim.x) {
    const int r = e / DV, d = e % DV;
    sG[e] = (q0 + r < p.Sq) ? p.dout[((size_t)bh * p.Sq + q0 + r) * DV + d] : 0.f;
  }
  float acc[16][4], lse[16], dl[16];
  int lo[16], hi[16];
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int i = q0 + warp * 16 + rr;
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[rr][t] = 0.f;
    lse[rr] = (i < p.Sq) ? p.lse[(size_t)bh * p.Sq + i] : -INFINITY;
    dl[rr] = (i < p.Sq) ? p.delta[(size_t)bh * p.Sq + i] : 0.f;
    row_interval(p.mask, i, p.Sq, p.Sk, lo[rr], hi[rr]);
  }
  TileWalk walk;
  int nslots;
  if (p.has_lists) {
    walk = make_walk(p.qmc, p.qmi, p.qfc, p.qfi, bh * p.nqb + q0 / p.sparse_m, p.nkb, p.sub_k, p.Sk);
    nslots = walk.nslots;
  } else {
    nslots = (p.Sk + 127) / 128;
  }
  for (int s = 0; s < nslots; ++s) {
    int kv0;
    bool masked;
    const bool ok = p.has_lists ? walk_slot(walk, s, p.mask, true, q0, p.Sq, p.Sk, &kv0, &masked)
                                : dense_slot(s, p.mask, true, q0, p.Sq, p.Sk, &kv0, &masked);
    if (!ok) continue;
    for (int c0 = kv0; c0 < kv0 + 128 && c0 < p.Sk; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * DQ; e += blockDim.x) {
        const int r = e / DQ, d = e % DQ;
        sK[r * (DQ + 1) + d] = (c0 + r < p.Sk) ? K[(size_t)(c0 + r) * DQ + d] : 0.f;
      }
      for (int e = threadIdx.x; e < kChunk * DV; e += blockDim.x) {
        const int r = e / DV, d = e % DV;
        sV[r * (DV + 1) + d] = (c0 + r < p.Sk) ? V[(size_t)(c0 + r) * DV + d] : 0.f;
      }
      __syncthreads();
      const int j = c0 + lane;
#pragma unroll 1
      for (int rr = 0; rr < 16; ++rr) {
        const int row = warp * 16 + rr, i = q0 + row;
        float dot = 0.f, dp = 0.f;
        for (int d = 0; d < DQ; ++d) dot = fmaf(sQ[row * DQ + d], sK[lane * (DQ + 1) + d], dot);
        for (int d = 0; d < DV; ++d) dp = fmaf(sG[row * DV + d], sV[lane * (DV + 1) + d], dp);
        float dcap;
        const float sc = simt_score(p, dot, i, j, kb, &dcap);
        const bool al = simt_allowed(p, bh, i, j, lo[rr], hi[rr], keep) && lse[rr] != -INFINITY;
        const float pj = al ? expf(sc - lse[rr]) : 0.f;
        const float ds = pj * (dp - dl[rr]) * dcap;
        for (int jj = 0; jj < kChunk; ++jj) {
          const float db = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int d = lane + 32 * t;
            if (d < DQ) acc[rr][t] = fmaf(db, sK[jj * (DQ + 1) + d], acc[rr][t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int i = q0 + warp * 16 + rr;
    if (i >= p.Sq) continue;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int d = lane + 32 * t;
      if (d < DQ) p.dq[((size_t)bh * p.Sq + i) * DQ + d] = acc[rr][t] * p.scale;
    }
  }
}

// dK, dV: CTA = (b, key/value head, 128-key tile), walking, for each query
// head of the group (GQA; one head without it), its backward list over query
// tiles; warp w owns keys 16 w .. 16 w + 15; lanes map to 32 query rows.
__global__ void __launch_bounds__(kSimtThreads) simt_dkdv_kernel(const SimtParams p) {
  extern __shared__ float sm[];
  const int DQ = p.Dqk, DV = p.Dv;
  float* sK = sm;                          // [128][DQ]
  float* sV = sK + 128 * DQ;               // [128][DV]
  float* sQ = sV + 128 * DV;               // [32][DQ + 1]
  float* sG = sQ + kChunk * (DQ + 1);      // [32][DV + 1]
  const int BHkv = p.B * p.Hkv;
  const int bkv = blockIdx.x % BHkv;
  const int k0 = (blockIdx.x / BHkv) * 128;
  const int bq0 = (bkv / p.Hkv) * p.H + (bkv % p.Hkv) * p.G;  // first query head of the group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < 128 * DQ; e += blockDim.x) {
    const int r = e / DQ, d = e % DQ;
    sK[e] = (k0 + r < p.Sk) ? p.k[((size_t)bkv * p.Sk + k0 + r) * DQ + d] : 0.f;
  }
  for (int e = threadIdx.x; e < 128 * DV; e += blockDim.x) {
    const int r = e / DV, d = e % DV;
    sV[e] = (k0 + r < p.Sk) ? p.v[((size_t)bkv * p.Sk + k0 + r) * DV + d] : 0.f;
  }
  float ak[16][4], av[16][4];
  float dbk[16];  // key-bias gradient: this lane's rows' sum of dS (before the softcap factor)
  int lo[16], hi[16];
  bool kept[16];
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    dbk[kk] = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) ak[kk][t] = av[kk][t] = 0.f;
    const int j = k0 + warp * 16 + kk;
    col_interval(p.mask, j, p.Sq, p.Sk, lo[kk], hi[kk]);
  }
  for (int g = 0; g < p.G; ++g) {
    const int bh = bq0 + g;  // query head
    const float* Q = p.q + (size_t)bh * p.Sq * DQ;
    const float* G = p.dout + (size_t)bh * p.Sq * DV;
    const float* kb = p.mask.key_bias ? p.mask.key_bias + (size_t)bh * p.Sk : nullptr;
    const uint32_t* keep = p.mask.keep ? p.mask.keep + (size_t)bh * p.mask.nkw : nullptr;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const int j = k0 + warp * 16 + kk;
      kept[kk] = (j < p.Sk) && (!keep || ((__ldg(keep + (j >> 5)) >> (j & 31)) & 1u));
    }
    TileWalk walk;
    int nslots;
    if (p.has_lists) {
      walk = make_walk(p.kmc, p.kmi, p.kfc, p.kfi, bh * p.nkb + k0 / p.sparse_n, p.nqb, p.sub_q, p.Sq);
      nslots = walk.nslots;
    } else {
      nslots = (p.Sq + 127) / 128;
    }
    for (int s = 0; s < nslots; ++s) {
      int qs;
      bool masked;
      const bool ok = p.has_lists ? walk_slot(walk, s, p.mask, false, k0, p.Sq, p.Sk, &qs, &masked)
                                  : dense_slot(s, p.mask, false, k0, p.Sq, p.Sk, &qs, &masked);
      if (!ok) continue;
      for (int r0 = qs; r0 < qs + 128 && r0 < p.Sq; r0 += kChunk) {
        __syncthreads();
        for (int e = threadIdx.x; e < kChunk * DQ; e += blockDim.x) {
          const int r = e / DQ, d = e % DQ;
          sQ[r * (DQ + 1) + d] = (r0 + r < p.Sq) ? Q[(size_t)(r0 + r) * DQ + d] : 0.f;
        }
        for (int e = threadIdx.x; e < kChunk * DV; e += blockDim.x) {
          const int r = e / DV, d = e % DV;
          sG[r * (DV + 1) + d] = (r0 + r < p.Sq) ? G[(size_t)(r0 + r) * DV + d] : 0.f;
        }
        __syncthreads();
        const int i = r0 + lane;
        const float lse = (i < p.Sq) ? p.lse[(size_t)bh * p.Sq + i] : -INFINITY;
        const float dl = (i < p.Sq) ? p.delta[(size_t)bh * p.Sq + i] : 0.f;
#pragma unroll 1
        for (int kk = 0; kk < 16; ++kk) {
          const int kr = warp * 16 + kk, j = k0 + kr;
          float dot = 0.f, dp = 0.f;
          for (int d = 0; d < DQ; ++d) dot = fmaf(sQ[lane * (DQ + 1) + d], sK[kr * DQ + d], dot);
          for (int d = 0; d < DV; ++d) dp = fmaf(sG[lane * (DV + 1) + d], sV[kr * DV + d], dp);
          float dcap;
          const float sc = simt_score(p, dot, i, j, kb, &dcap);
          const bool al = kept[kk] && i >= lo[kk] && i <= hi[kk] && i < p.Sq && lse != -INFINITY &&
                          (!p.mask.table || ((__ldg(table_row(p.mask, bh, p.Sq, i) + (j >> 5)) >> (j & 31)) & 1u));
          const float pj = al ? expf(sc - lse) : 0.f;
          const float ds0 = pj * (dp - dl);
          dbk[kk] += ds0;
          const float ds = ds0 * dcap;
          for (int ii = 0; ii < kChunk; ++ii) {
            const float pb = __shfl_sync(0xffffffffu, pj, ii);
            const float db = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int d = lane + 32 * t;
              if (d < DV) av[kk][t] = fmaf(pb, sG[ii * (DV + 1) + d], av[kk][t]);
              if (d < DQ) ak[kk][t] = fmaf(db, sQ[ii * (DQ + 1) + d], ak[kk][t]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const int j = k0 + warp * 16 + kk;
    float db = dbk[kk];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) db += __shfl_xor_sync(0xffffffffu, db, off);
    if (j >= p.Sk) continue;
    // key-bias gradient: one query head per key/value head (the host rejects it with GQA)
    if (p.dbias && lane == 0) p.dbias[(size_t)bq0 * p.Sk + j] = db;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int d = lane + 32 * t;
      if (d < DV) p.dv[((size_t)bkv * p.Sk + j) * DV + d] = av[kk][t];
      if (d < DQ) p.dk[((size_t)bkv * p.Sk + j) * DQ + d] = ak[kk][t] * p.scale;
    }
  }
}

static void fill_simt(SimtParams& prm, const Shape& s, float scale, const HostMask& m) {
  memset(&prm, 0, sizeof(prm));
  prm.B = s.B;
  prm.H = s.H;
  prm.Sq = s.Sq;
  prm.Sk = s.Sk;
  prm.Dqk = s.Dqk;
  prm.Dv = s.Dv;
  prm.Hkv = s.Hkv;
  prm.G = s.H / s.Hkv;
  prm.scale = scale;
  prm.softcap = m.softcap;
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
  prm.has_lists = m.has_lists;
  if (m.has_lists) {
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
}

static int set_smem(const void* fn, size_t bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess
             ? GBATTN_OK
             : GBATTN_ERR_CUDA;
}

int fwd_fp32_launch(const Shape& s, const float* q, const float* k, const float* v, float scale, const HostMask& m,
                    float* o, float* lse, cudaStream_t st) {
  SimtParams prm;
  fill_simt(prm, s, scale, m);
  prm.q = q;
  prm.k = k;
  prm.v = v;
  prm.out = o;
  prm.lse_out = lse;
  const size_t smem = sizeof(float) * (128 * s.Dqk + kChunk * (s.Dqk + 1) + kChunk * s.Dv);
  if (set_smem((const void*)simt_fwd_kernel, smem)) return GBATTN_ERR_CUDA;
  const int grid = ((s.Sq + 127) / 128) * s.B * s.H;
  simt_fwd_kernel<<<grid, kSimtThreads, smem, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int bwd_fp32_launch(const Shape& s, const float* q, const float* k, const float* v, const float* o, const float* dout,
                    const float* lse, float scale, const HostMask& m, float* dq, float* dk, float* dv,
                    float* dkey_bias, void* ws, cudaStream_t st) {
  SimtParams prm;
  fill_simt(prm, s, scale, m);
  prm.q = q;
  prm.k = k;
  prm.v = v;
  prm.o = o;
  prm.dout = dout;
  prm.lse = lse;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.dbias = dkey_bias;
  const size_t BH = (size_t)s.B * s.H;
  prm.delta = reinterpret_cast<float*>(ws);
  const long long rows = (long long)BH * s.Sq;
  simt_delta_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  const size_t smq = sizeof(float) * (128 * s.Dqk + 128 * s.Dv + kChunk * (s.Dqk + 1) + kChunk * (s.Dv + 1));
  if (set_smem((const void*)simt_dq_kernel, smq)) return GBATTN_ERR_CUDA;
  simt_dq_kernel<<<(unsigned)(((s.Sq + 127) / 128) * BH), kSimtThreads, smq, st>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  const size_t smk = sizeof(float) * (128 * s.Dqk + 128 * s.Dv + kChunk * (s.Dqk + 1) + kChunk * (s.Dv + 1));
  if (set_smem((const void*)simt_dkdv_kernel, smk)) return GBATTN_ERR_CUDA;
  simt_dkdv_kernel<<<(unsigned)(((s.Sk + 127) / 128) * s.B * s.Hkv), kSimtThreads, smk, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

GB_DEFINE_ERROR_READER(simt_take_error)

}  // namespace gb
