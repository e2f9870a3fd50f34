// decode.cu - split-KV forward for decode shapes, and the split combine.
//
// "Optimize Flash Dynamic Mask Attention Kernel Configurations" simplifies the
// split-KV forward path and tests 1/2/4/8/16 splits; it also notes that
// Q = 1 / very long K is memory-bound. Here each CTA = (b, h, query row,
// split) streams its contiguous K/V key range once from HBM with 1-D bulk
// copies (cp.async.bulk) into a 4-stage shared-memory ring; 8 compute warps
// read 16-byte vectors from it. Each warp keeps its own running max / sum /
// output over its keys (online softmax); the warps are merged at the end and
// the split partials are merged by a combine kernel using the rule of the
// POPCORNBENCH "Kimi-K2.6 l1_p97" trace: m = max_s m_s, weights exp(m_s - m).
//
// The key/value rows come from a dense cache [B, Hkv, Sk, D] or from a paged
// cache (pages of page_size keys of one key/value head, [num_pages, Hkv,
// page_size, D], mapped per sequence by a page table), optionally with a
// per-sequence key count. Query heads share key/value heads in groups of
// G = H / Hkv (GQA); the G CTAs of a group stream the same rows close in time,
// so the repeats are served by L2.
#include <mutex>

#include "kernels.h"
#include "mask.cuh"

namespace gb {

constexpr int kDecWarps = 8;                 // compute warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);
constexpr int kDecChunk = 64;                // keys per stage
constexpr int kDecStages = 4;

struct DecParams {
  const __nv_bfloat16 *q, *k, *v;
  __nv_bfloat16* o;
  float* lse;
  float* o_part;     // [n][BH][Sq][D]
  float* lse_part;   // [n][BH][Sq]
  int BH, Sq, Sk, nsplit, causal;
  int H, Hkv, G;     // query heads, key/value heads, H / Hkv
  const int32_t* seqlens;     // [B] keys per sequence, or nullptr (all Sk)
  const int32_t* page_table;  // [B][max_pages], or nullptr (dense cache)
  int page_size, max_pages, num_pages;
  float scale_log2;
  unsigned long long wait_ns;  // time limit of every wait (0 = kWaitLimitNs)
};

// Address of the key/value row `key` of sequence b, key/value head hkv.
template <int D>
__device__ __forceinline__ size_t kv_row(const DecParams& p, int b, int hkv, int key) {
  if (!p.page_table) return ((size_t)(b * p.Hkv + hkv) * p.Sk + key) * D;
  int page = __ldg(p.page_table + (size_t)b * p.max_pages + key / p.page_size);
  if (page < 0 || page >= p.num_pages) {
    raise_dev_error(GBATTN_ERR_BLOCKS);  // read page 0 instead; the output is invalid
    page = 0;
  }
  return ((size_t)(page * p.Hkv + hkv) * p.page_size + key % p.page_size) * D;
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1) splitkv_kernel(const DecParams p) {
  constexpr int ROWB = D * 2;                       // bytes per key row
  constexpr int CHB = kDecChunk * ROWB;             // bytes per K (or V) chunk
  constexpr int EPL = D / 32;                       // V elements per lane (PV phase)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* sK = base;
  uint8_t* sV = sK + kDecStages * CHB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sV + kDecStages * CHB);
  uint64_t* empty = full + kDecStages;
  float* red = reinterpret_cast<float*>(empty + kDecStages);  // [kDecWarps][D + 2]
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(red + kDecWarps * (D + 2)), p.wait_ns);

  const int split = blockIdx.x % p.nsplit;
  const int rowid = blockIdx.x / p.nsplit;  // bh * Sq + i
  const int bh = rowid / p.Sq, i = rowid % p.Sq;
  const int b = bh / p.H, hkv = (bh % p.H) / p.G;
  int skb = p.Sk;  // keys of this sequence
  if (p.seqlens) {
    skb = __ldg(p.seqlens + b);
    const int cap = p.page_table ? p.max_pages * p.page_size : p.Sk;
    if (skb < 0 || skb > cap) {
      if (threadIdx.x == 0) raise_dev_error(GBATTN_ERR_BLOCKS);
      skb = max(0, min(skb, cap));
    }
  }
  // split s covers keys [s L, (s + 1) L), L = ceil(keys / n) rounded up to 128
  const int per = ((skb + p.nsplit - 1) / p.nsplit + 127) / 128 * 128;
  int kb = split * per;
  int ke = min(kb + per, skb);
  if (p.causal) ke = min(ke, i + (skb - p.Sq) + 1);
  const int nkeys = max(0, ke - kb);
  const int nchunks = (nkeys + kDecChunk - 1) / kDecChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();


  if (warp == kDecWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kDecStages;
        if (c >= kDecStages && !mbar_wait(empty + s, ((c / kDecStages) + 1) & 1, abort_flag)) break;
        const int rows = min(kDecChunk, nkeys - c * kDecChunk);
        const uint32_t bytes = (uint32_t)rows * ROWB;
        // a chunk never crosses a page: kb is a multiple of 128 and pages hold a
        // multiple of 64 keys
        const size_t off = kv_row<D>(p, b, hkv, kb + c * kDecChunk);
        mbar_expect_tx(full + s, 2 * bytes);
        bulk_load(sK + s * CHB, p.k + off, bytes, full + s);
        bulk_load(sV + s * CHB, p.v + off, bytes, full + s);
        ++issued;
      }
      if (*abort_flag)
        for (int c = (issued > kDecStages ? issued - kDecStages : 0); c < issued; ++c)
          mbar_drain(full + c % kDecStages, (c / kDecStages) & 1, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int g = lane >> 3, sub = lane & 7;  // 4 groups of 8 lanes, one key per group
    // q slice of this lane for the score phase: elements [64 h + 8 sub, +8)
    float qv[D / 8];
    const __nv_bfloat16* qrow = p.q + ((size_t)bh * p.Sq + i) * D;
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      const uint4 raw = *reinterpret_cast<const uint4*>(qrow + h * 64 + sub * 8);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(b2[e]);
        qv[h * 8 + 2 * e] = f.x * p.scale_log2;
        qv[h * 8 + 2 * e + 1] = f.y * p.scale_log2;
      }
    }
    float m = -INFINITY, l = 0.f;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kDecStages;
      ok = mbar_wait(full + s, (c / kDecStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const int rows = min(kDecChunk, nkeys - c * kDecChunk);
      const uint8_t* kc = sK + s * CHB;
      const uint8_t* vc = sV + s * CHB;
      // scores of this warp's 8 keys: key (warp * 8 + it * 4 + g)
      float sc[2];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int key = warp * 8 + it * 4 + g;
        float dot = 0.f;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          const uint4 raw = *reinterpret_cast<const uint4*>(kc + key * ROWB + h * 128 + sub * 16);
          const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b2[e]);
            dot = fmaf(f.x, qv[h * 8 + 2 * e], dot);
            dot = fmaf(f.y, qv[h * 8 + 2 * e + 1], dot);
          }
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        dot += __shfl_xor_sync(0xffffffffu, dot, 4);
        sc[it] = (key < rows) ? dot : -INFINITY;
      }
      float mc = fmaxf(sc[0], sc[1]);
      mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 8));
      mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 16));
      const float mn = fmaxf(m, mc);
      const float msafe = (mn == -INFINITY) ? 0.f : mn;
      const float alpha = ex2(m - msafe);  // m = -inf -> 0
      float pr[2];
      pr[0] = ex2(sc[0] - msafe);
      pr[1] = ex2(sc[1] - msafe);
      float ls = pr[0] + pr[1];
      ls += __shfl_xor_sync(0xffffffffu, ls, 8);
      ls += __shfl_xor_sync(0xffffffffu, ls, 16);
      l = l * alpha + ls;
      m = mn;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
      // O += sum over the 8 keys of p_key * v_key; lane owns EPL dims
#pragma unroll
      for (int it = 0; it < 2; ++it) {
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const float pk = __shfl_sync(0xffffffffu, pr[it], gg * 8);
          const int key = warp * 8 + it * 4 + gg;
          if (key >= rows) continue;  // stale smem beyond the chunk end
          if constexpr (EPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(vc + key * ROWB + lane * 8);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
            const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
            acc[0] = fmaf(pk, f0.x, acc[0]);
            acc[1] = fmaf(pk, f0.y, acc[1]);
            acc[2] = fmaf(pk, f1.x, acc[2]);
            acc[3] = fmaf(pk, f1.y, acc[3]);
          } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(vc + key * ROWB + lane * 4);
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw));
            acc[0] = fmaf(pk, f0.x, acc[0]);
            acc[1] = fmaf(pk, f0.y, acc[1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
    // publish this warp's (m, l, acc) for the merge
    float* rw = red + warp * (D + 2);
#pragma unroll
    for (int e = 0; e < EPL; ++e) rw[lane * EPL + e] = acc[e];
    if (lane == 0) {
      rw[D] = m;
      rw[D + 1] = l;
    }
  }
  __syncthreads();
  if (*abort_flag) return;
  // merge the warps (threads 0..D-1, one output element each)
  if (threadIdx.x < D) {
    const int d = threadIdx.x;
    float mx = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, red[w * (D + 2) + D]);
    float lt = 0.f, ot = 0.f;
    if (mx != -INFINITY) {
      for (int w = 0; w < kDecWarps; ++w) {
        const float wgt = ex2(red[w * (D + 2) + D] - mx);
        lt += wgt * red[w * (D + 2) + D + 1];
        ot += wgt * red[w * (D + 2) + d];
      }
    }
    const bool live = lt > 0.f;
    const float val = live ? ot / lt : 0.f;
    const float lse_nat = live ? (mx + __log2f(lt)) * kLn2 : -INFINITY;
    if (p.nsplit == 1) {
      p.o[(size_t)rowid * D + d] = __float2bfloat16_rn(val);
      if (d == 0 && p.lse) p.lse[rowid] = lse_nat;
    } else {
      const size_t prow = (size_t)split * p.BH * p.Sq + rowid;
      p.o_part[prow * D + d] = val;
      if (d == 0) p.lse_part[prow] = lse_nat;
    }
  }
}

// Grouped decode (GQA, pack-GQA): CTA = (b, key/value head, split, chunk of
// RC = 4 RPG query rows of the group). The G query heads of a key/value head
// (G x Sq rows, contiguous in Q, O and LSE) share every key/value row, so the
// CTA streams each 64-key chunk once and all its rows use it: the four lane
// groups of a warp take different rows of the same key, their shared-memory
// reads of K and V are broadcasts, and each lane keeps 1/8 of the head dim of
// its rows (scores reduced over the 8 lanes of a group). Each warp keeps its
// own online softmax over its 8 keys of every chunk; the warps are merged at
// the end and the splits by combine_kernel, as in splitkv_kernel. Nine warps
// put three on one SM sub-partition, so a thread has at most 168 registers:
// 16 rows per CTA fit at D = 64, 8 rows at D = 128.
template <int D, int RPG>
__global__ void __launch_bounds__(kDecThreads, 1) splitkv_group_kernel(const DecParams p, int nrch) {
  constexpr int ROWB = D * 2;
  constexpr int CHB = kDecChunk * ROWB;
  constexpr int RC = 4 * RPG;     // query rows of this CTA
  constexpr int SL = D / 8;       // head-dim elements of a lane: D/64 slabs of 8
  constexpr int NS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* sK = base;
  uint8_t* sV = sK + kDecStages * CHB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sV + kDecStages * CHB);
  uint64_t* empty = full + kDecStages;
  float* red = reinterpret_cast<float*>(empty + kDecStages);  // [kDecWarps][RC][D + 2]
  const WaitCtl abort_flag = wait_ctl(reinterpret_cast<volatile int*>(red + kDecWarps * RC * (D + 2)), p.wait_ns);

  const int split = blockIdx.x % p.nsplit;
  const int rest = blockIdx.x / p.nsplit;
  const int rch = rest % nrch;
  const int bkv = rest / nrch;
  const int b = bkv / p.Hkv, hkv = bkv % p.Hkv;
  const int R = p.G * p.Sq;                                 // query rows of the group
  const int row0 = (b * p.H + hkv * p.G) * p.Sq;            // first row id of the group
  const int rc0 = rch * RC;                                 // first group row of this CTA
  int skb = p.Sk;
  if (p.seqlens) {
    skb = __ldg(p.seqlens + b);
    const int cap = p.page_table ? p.max_pages * p.page_size : p.Sk;
    if (skb < 0 || skb > cap) {
      if (threadIdx.x == 0) raise_dev_error(GBATTN_ERR_BLOCKS);
      skb = max(0, min(skb, cap));
    }
  }
  const int per = ((skb + p.nsplit - 1) / p.nsplit + 127) / 128 * 128;
  const int kb = split * per;
  const int ke = min(kb + per, skb);
  const int nkeys = max(0, ke - kb);
  const int nchunks = (nkeys + kDecChunk - 1) / kDecChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kDecStages;
        if (c >= kDecStages && !mbar_wait(empty + s, ((c / kDecStages) + 1) & 1, abort_flag)) break;
        const int rows = min(kDecChunk, nkeys - c * kDecChunk);
        const uint32_t bytes = (uint32_t)rows * ROWB;
        const size_t off = kv_row<D>(p, b, hkv, kb + c * kDecChunk);
        mbar_expect_tx(full + s, 2 * bytes);
        bulk_load(sK + s * CHB, p.k + off, bytes, full + s);
        bulk_load(sV + s * CHB, p.v + off, bytes, full + s);
        ++issued;
      }
      if (*abort_flag)
        for (int c = (issued > kDecStages ? issued - kDecStages : 0); c < issued; ++c)
          mbar_drain(full + c % kDecStages, (c / kDecStages) & 1, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int g = lane >> 3, sub = lane & 7;  // group: rows g*RPG.., sub: head-dim slice
    float qv[RPG][SL];
    int lim[RPG];  // last allowed key index of each row (-1: padding row)
#pragma unroll
    for (int t = 0; t < RPG; ++t) {
      const int r = rc0 + g * RPG + t;
      lim[t] = -1;
#pragma unroll
      for (int e = 0; e < SL; ++e) qv[t][e] = 0.f;
      if (r < R) {
        const int i = r % p.Sq;
        lim[t] = p.causal ? i + (skb - p.Sq) : skb - 1;
        const __nv_bfloat16* qrow = p.q + (size_t)(row0 + r) * D;
#pragma unroll
        for (int h = 0; h < NS; ++h) {
          const uint4 raw = *reinterpret_cast<const uint4*>(qrow + h * 64 + sub * 8);
          const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b2[e]);
            qv[t][h * 8 + 2 * e] = f.x * p.scale_log2;
            qv[t][h * 8 + 2 * e + 1] = f.y * p.scale_log2;
          }
        }
      }
    }
    float m[RPG], l[RPG], acc[RPG][SL];
#pragma unroll
    for (int t = 0; t < RPG; ++t) {
      m[t] = -INFINITY;
      l[t] = 0.f;
#pragma unroll
      for (int e = 0; e < SL; ++e) acc[t][e] = 0.f;
    }
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kDecStages;
      ok = mbar_wait(full + s, (c / kDecStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const int rows = min(kDecChunk, nkeys - c * kDecChunk);
      const uint8_t* kc = sK + s * CHB;
      const uint8_t* vc = sV + s * CHB;
      const int key0 = kb + c * kDecChunk + warp * 8;  // index of this warp's first key
      float sc[RPG][8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int key = warp * 8 + k;
        float kf[SL];
        if (key < rows) {
#pragma unroll
          for (int h = 0; h < NS; ++h) {
            const uint4 raw = *reinterpret_cast<const uint4*>(kc + key * ROWB + h * 128 + sub * 16);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(b2[e]);
              kf[h * 8 + 2 * e] = f.x;
              kf[h * 8 + 2 * e + 1] = f.y;
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < SL; ++e) kf[e] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < RPG; ++t) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < SL; ++e) dot = fmaf(kf[e], qv[t][e], dot);
          dot += __shfl_xor_sync(0xffffffffu, dot, 1);
          dot += __shfl_xor_sync(0xffffffffu, dot, 2);
          dot += __shfl_xor_sync(0xffffffffu, dot, 4);
          sc[t][k] = (key < rows && key0 + k <= lim[t]) ? dot : -INFINITY;
        }
      }
      // probabilities in place of the scores
#pragma unroll
      for (int t = 0; t < RPG; ++t) {
        float mc = sc[t][0];
#pragma unroll
        for (int k = 1; k < 8; ++k) mc = fmaxf(mc, sc[t][k]);
        const float mn = fmaxf(m[t], mc);
        const float msafe = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = ex2(m[t] - msafe);  // m = -inf -> 0
        float ls = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          sc[t][k] = ex2(sc[t][k] - msafe);
          ls += sc[t][k];
        }
        l[t] = l[t] * alpha + ls;
        m[t] = mn;
#pragma unroll
        for (int e = 0; e < SL; ++e) acc[t][e] *= alpha;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int key = warp * 8 + k;
        if (key >= rows) continue;  // stale shared memory beyond the chunk end
        float vf[SL];
#pragma unroll
        for (int h = 0; h < NS; ++h) {
          const uint4 raw = *reinterpret_cast<const uint4*>(vc + key * ROWB + h * 128 + sub * 16);
          const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b2[e]);
            vf[h * 8 + 2 * e] = f.x;
            vf[h * 8 + 2 * e + 1] = f.y;
          }
        }
#pragma unroll
        for (int t = 0; t < RPG; ++t)
#pragma unroll
          for (int e = 0; e < SL; ++e) acc[t][e] = fmaf(sc[t][k], vf[e], acc[t][e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
    // publish this warp's (m, l, acc) of each row for the merge
#pragma unroll
    for (int t = 0; t < RPG; ++t) {
      float* rw = red + (warp * RC + g * RPG + t) * (D + 2);
#pragma unroll
      for (int h = 0; h < NS; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) rw[h * 64 + sub * 8 + e] = acc[t][h * 8 + e];
      if (sub == 0) {
        rw[D] = m[t];
        rw[D + 1] = l[t];
      }
    }
  }
  __syncthreads();
  if (*abort_flag) return;
  // merge the warps: one output element per thread and step
  for (int idx = threadIdx.x; idx < RC * D; idx += blockDim.x) {
    const int rr = idx / D, d = idx % D;
    const int r = rc0 + rr;
    if (r >= R) continue;
    float mx = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, red[(w * RC + rr) * (D + 2) + D]);
    float lt = 0.f, ot = 0.f;
    if (mx != -INFINITY) {
      for (int w = 0; w < kDecWarps; ++w) {
        const float* rw = red + (w * RC + rr) * (D + 2);
        const float wgt = ex2(rw[D] - mx);
        lt += wgt * rw[D + 1];
        ot += wgt * rw[d];
      }
    }
    const bool live = lt > 0.f;
    const float val = live ? ot / lt : 0.f;
    const float lse_nat = live ? (mx + __log2f(lt)) * kLn2 : -INFINITY;
    const int rowid = row0 + r;
    if (p.nsplit == 1) {
      p.o[(size_t)rowid * D + d] = __float2bfloat16_rn(val);
      if (d == 0 && p.lse) p.lse[rowid] = lse_nat;
    } else {
      const size_t prow = (size_t)split * p.BH * p.Sq + rowid;
      p.o_part[prow * D + d] = val;
      if (d == 0) p.lse_part[prow] = lse_nat;
    }
  }
}

// One warp per (b, h, query row): merge the split partials.
template <int D>
__global__ void combine_kernel(const DecParams p) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.BH * p.Sq;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < p.nsplit; ++s) mx = fmaxf(mx, p.lse_part[s * rows + row]);
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
  float tot = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < p.nsplit; ++s) {
      const float ls = p.lse_part[s * rows + row];
      const float w = (ls == -INFINITY) ? 0.f : __expf(ls - mx);
      tot += w;
      const float* op = p.o_part + (s * rows + row) * D;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(w, op[lane + 32 * e], acc[e]);
    }
  }
  const bool live = tot > 0.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e)
    p.o[row * D + lane + 32 * e] = __float2bfloat16_rn(live ? acc[e] / tot : 0.f);
  if (lane == 0 && p.lse) p.lse[row] = live ? mx + __logf(tot) : -INFINITY;
}

template <int D, int RPG>
static int launch_group(const DecParams& prm, cudaStream_t st) {
  constexpr int CHB = kDecChunk * D * 2;
  constexpr int RC = 4 * RPG;
  constexpr int SMEM = 128 + 2 * kDecStages * CHB + 2 * kDecStages * 8 + kDecWarps * RC * (D + 2) * 4 + 16;
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(splitkv_group_kernel<D, RPG>, SMEM, attr)) return GBATTN_ERR_CUDA;
  const int R = prm.G * prm.Sq;
  const int nrch = (R + RC - 1) / RC;
  const long long grid = (long long)(prm.BH / prm.G) * nrch * prm.nsplit;
  if (grid >= (1ll << 31)) return GBATTN_ERR_ARG;
  splitkv_group_kernel<D, RPG><<<(unsigned)grid, kDecThreads, SMEM, st>>>(prm, nrch);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

template <int D>
static int launch_dec(const DecParams& prm, cudaStream_t st) {
  constexpr int CHB = kDecChunk * D * 2;
  constexpr int SMEM = 128 + 2 * kDecStages * CHB + 2 * kDecStages * 8 + kDecWarps * (D + 2) * 4 + 16;
  static std::atomic<unsigned long long> attr{0};
  if (ensure_smem(splitkv_kernel<D>, SMEM, attr)) return GBATTN_ERR_CUDA;
  const int R = prm.G * prm.Sq;  // query rows per key/value head
  if (prm.G > 1 && R >= 4) {
    // query heads share key/value heads: one CTA streams each chunk for up to 8 (D=128) or 16 (D=64) rows
    constexpr int RPG_MAX = D <= 64 ? 4 : 2;
    const int rc = R <= 4 ? launch_group<D, 1>(prm, st) : (R <= 8 || RPG_MAX == 2) ? launch_group<D, 2>(prm, st)
                                                                                   : launch_group<D, RPG_MAX>(prm, st);
    if (rc != GBATTN_OK) return rc;
  } else {
    const long long grid = (long long)prm.BH * prm.Sq * prm.nsplit;
    if (grid >= (1ll << 31)) return GBATTN_ERR_ARG;
    splitkv_kernel<D><<<(unsigned)grid, kDecThreads, SMEM, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  }
  if (prm.nsplit > 1) {
    const long long rows = (long long)prm.BH * prm.Sq;
    combine_kernel<D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  }
  return GBATTN_OK;
}

int splitkv_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                   int num_splits, void* o, float* lse, void* ws, cudaStream_t st, const PagedKV* paged) {
  DecParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.H = s.H;
  prm.Hkv = s.Hkv;
  prm.G = s.H / s.Hkv;
  if (paged) {
    prm.seqlens = paged->seqlens;
    prm.page_table = paged->page_table;
    prm.page_size = paged->page_size;
    prm.max_pages = paged->max_pages;
    prm.num_pages = paged->num_pages;
  }
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.BH = s.B * s.H;
  prm.Sq = s.Sq;
  prm.Sk = s.Sk;
  prm.nsplit = num_splits;
  prm.causal = causal;
  prm.scale_log2 = scale * kLog2e;
  if (num_splits > 1) {
    const size_t rows = (size_t)num_splits * prm.BH * s.Sq;
    prm.o_part = static_cast<float*>(ws);
    prm.lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(rows * s.Dv * sizeof(float), 256));
  }
  if (prm.G > 1 && (!paged || !paged->page_table || paged->page_size % 128 == 0)) {
    // grouped query heads: the group's rows packed into 128-row tiles of the
    // tensor-core forward kernel, one CTA per key/value tile range (a paged
    // pool qualifies when a 128-key tile never crosses a page)
    const int rc = fwd_packed_decode_launch(s, q, k, v, scale, causal, num_splits, o, lse, prm.o_part, prm.lse_part,
                                            paged, st);
    if (rc != GBATTN_OK || num_splits == 1) return rc;
    const long long rows = (long long)prm.BH * prm.Sq;
    if (s.Dqk == 128) combine_kernel<128><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(prm);
    else combine_kernel<64><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(prm);
    return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
  }
  if (s.Dqk == 128) return launch_dec<128>(prm, st);
  if (s.Dqk == 64) return launch_dec<64>(prm, st);
  return GBATTN_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------------------
// Allocation-free split-KV: the split partials live in this file-scope array
// (GBATTN_NOALLOC_SCRATCH_BYTES), for callers that may not allocate device
// memory. Host code cannot use the array's name as a device address; the
// address is looked up once per device with that device current. Nothing in
// the array needs to start at zero: every split writes its whole partial
// (empty splits write LSE = -inf and zeros). Calls that overlap on the GPU
// share the array and race.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[GBATTN_NOALLOC_SCRATCH_BYTES];

static void* noalloc_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

int splitkv_noalloc_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                           int num_splits, size_t workspace_bytes, void* o, float* lse, cudaStream_t st) {
  if (workspace_bytes > (size_t)GBATTN_NOALLOC_SCRATCH_BYTES) return GBATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (num_splits > 1) {
    scratch = noalloc_scratch_address();
    if (!scratch) return GBATTN_ERR_CUDA;
  }
  return splitkv_launch(s, q, k, v, scale, causal, num_splits, o, lse, scratch, st, nullptr);
}

GB_DEFINE_ERROR_READER(decode_take_error)

}  // namespace gb
