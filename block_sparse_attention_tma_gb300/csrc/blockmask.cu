// blockmask.cu - build_block_mask: the dynamic keep set (top-k per head) and
// the forward / backward block-sparse lists.
//
// "Enable 2CTA for SM100 block-sparse backward" builds, from one mask
// predicate, per-q-block lists of kv-blocks for the forward and per-kv-block
// lists of q-blocks for the backward, each split into blocks that need the
// element mask and blocks that are fully allowed. The dynamic mask of
// "Optimize Flash Dynamic Mask Attention Kernel Configurations" keeps, per
// (b, h), the top-k keys ranked by the additive key bias (ties: lower index).
//
// All integer work; the top-k compares fp32 biases through an
// order-preserving 32-bit key, so the result is exact.
#include "kernels.h"
#include "mask.cuh"

namespace gb {

// Order-preserving map float -> uint32 (larger float -> larger key); -0 and +0
// map to the same key so that they tie, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (x == 0.f) x = 0.f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 1024;

// One CTA per (b, h). Radix select (8-bit digits, most significant first)
// finds the k-th largest key T and how many keys equal to T are kept; then
// keys > T are kept, and keys == T in ascending index order until the quota
// is met.
__global__ void __launch_bounds__(kTopkThreads) topk_keep_kernel(const float* __restrict__ bias, int Sk, int k,
                                                                 uint32_t* __restrict__ keep, int nkw) {
  const int bh = blockIdx.x;
  const float* b = bias + (size_t)bh * Sk;
  uint32_t* kw = keep + (size_t)bh * nkw;
  __shared__ unsigned int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int warp_sums[kTopkThreads / 32];
  __shared__ int s_carry;
  const int tid = threadIdx.x;

  if (k >= Sk || k <= 0) {
    const uint32_t fill = k > 0 ? 0xffffffffu : 0u;
    for (int w = tid; w < nkw; w += blockDim.x) {
      uint32_t v = fill;
      const int rem = Sk - w * 32;
      if (rem < 32) v &= (rem <= 0) ? 0u : ((1u << rem) - 1u);
      kw[w] = v;
    }
    return;
  }

  uint32_t prefix = 0, pmask = 0;
  int need = k;
  for (int d = 3; d >= 0; --d) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int sh = 8 * d;
    for (int j = tid; j < Sk; j += blockDim.x) {
      const uint32_t key = order_key(b[j]);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      int acc = 0, bin = 255;
      for (; bin >= 0; --bin) {
        if (acc + (int)hist[bin] >= need) break;
        acc += hist[bin];
      }
      s_need = need - acc;
      s_prefix = prefix | ((uint32_t)bin << sh);
    }
    __syncthreads();
    need = s_need;
    prefix = s_prefix;
    pmask |= 255u << sh;
    __syncthreads();
  }
  const uint32_t T = prefix;
  // keep keys > T, and the first `need` keys == T by ascending index
  if (tid == 0) s_carry = 0;
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < Sk; base += blockDim.x) {
    const int j = base + tid;
    uint32_t key = 0;
    if (j < Sk) key = order_key(b[j]);
    const bool tie = (j < Sk) && key == T;
    const unsigned tb = __ballot_sync(0xffffffffu, tie);
    const int before_in_warp = __popc(tb & ((1u << lane) - 1u));
    if (lane == 0) warp_sums[warp] = __popc(tb);
    __syncthreads();
    int before_warps = 0;
    for (int w = 0; w < warp; ++w) before_warps += warp_sums[w];
    const int rank = s_carry + before_warps + before_in_warp;
    const bool kept = (j < Sk) && (key > T || (tie && rank < need));
    const unsigned kb = __ballot_sync(0xffffffffu, kept);
    if (lane == 0 && (base + warp * 32) < Sk) kw[(base + warp * 32) >> 5] = kb;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += warp_sums[w];
      s_carry += tot;
    }
    __syncthreads();
  }
}

// One CTA per (b, h): the kept-key index list, i.e. the indices of the set
// bits of the keep mask in ascending order, then 0 up to Sk. A block-wide
// exclusive scan of the kept flags gives each kept key its slot.
__global__ void __launch_bounds__(kTopkThreads) keep_index_kernel(const uint32_t* __restrict__ keep, int Sk,
                                                                  int nkw, int32_t* __restrict__ idx) {
  const int bh = blockIdx.x;
  const uint32_t* kw = keep + (size_t)bh * nkw;
  int32_t* out = idx + (size_t)bh * Sk;
  __shared__ int warp_sums[kTopkThreads / 32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < Sk; base += blockDim.x) {
    const int j = base + tid;
    const bool kept = j < Sk && ((__ldg(kw + (j >> 5)) >> (j & 31)) & 1u);
    const unsigned b = __ballot_sync(0xffffffffu, kept);
    if (lane == 0) warp_sums[warp] = __popc(b);
    __syncthreads();
    int before = s_carry;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    if (kept) out[before + __popc(b & ((1u << lane) - 1u))] = j;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += warp_sums[w];
      s_carry += tot;
    }
    __syncthreads();
  }
  for (int t = s_carry + tid; t < Sk; t += blockDim.x) out[t] = 0;
}

struct ListArgs {
  MaskParams mask;
  int Sq, Sk, sm, sn, nqb, nkb, BH;
  int32_t *q_mask_cnt, *q_mask_idx, *q_full_cnt, *q_full_idx;
  int32_t *k_mask_cnt, *k_mask_idx, *k_full_cnt, *k_full_idx;
};

// Number of allowed pairs of sparse block (r, c), summed by the 32 lanes of
// a warp over the block's rows; every lane gets the total.
__device__ long long block_pairs(const ListArgs& a, int bh, int r, int c) {
  const int r0 = r * a.sm, r1 = min(r0 + a.sm, a.Sq);
  const int c0 = c * a.sn, c1 = min(c0 + a.sn, a.Sk);
  const int lane = threadIdx.x & 31;
  long long cnt = 0;
  const uint32_t* keep = a.mask.keep ? a.mask.keep + (size_t)bh * a.mask.nkw : nullptr;
  for (int i = r0 + lane; i < r1; i += 32) {
    int lo, hi;
    row_interval(a.mask, i, a.Sq, a.Sk, lo, hi);
    const int s = max(lo, c0), e = min(hi, c1 - 1);
    if (e < s) continue;
    // dynamic: the head's keep bits; element table: this row's bits
    const uint32_t* bitsrc = a.mask.table ? table_row(a.mask, bh, a.Sq, i) : keep;
    if (bitsrc) {
      for (int w = s >> 5; w <= (e >> 5); ++w) {
        uint32_t bits = __ldg(bitsrc + w);
        const int wb = w << 5;
        if (s > wb) bits &= ~((1u << (s - wb)) - 1u);
        if (e < wb + 31) bits &= (1u << (e - wb + 1)) - 1u;
        cnt += __popc(bits);
      }
    } else {
      cnt += e - s + 1;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt;
}

// 0 = absent, 1 = needs the element mask, 2 = full.
__device__ int block_class(const ListArgs& a, int bh, int r, int c) {
  const long long n = block_pairs(a, bh, r, c);
  if (n == 0) return 0;
  const int rows = min(a.sm, a.Sq - r * a.sm), cols = min(a.sn, a.Sk - c * a.sn);
  if (rows == a.sm && cols == a.sn && n == (long long)a.sm * a.sn) return 2;
  return 1;
}

constexpr int kListWarps = 8, kListChunk = 256;

// One CTA per (b, h, fixed block): the list of the streamed blocks of that
// block row (forward: fixed = q-block, streamed = k-blocks) or column
// (backward: fixed = k-block, streamed = q-blocks). The streamed blocks are
// taken in chunks of 256; each of the 8 warps classifies every 8th block of
// the chunk (one warp-collective pair count per block), then the 256 threads
// compact the chunk's mask and full entries in ascending order with a
// block-wide scan. Tail entries are 0.
template <bool FWD>
__global__ void __launch_bounds__(kListWarps * 32) lists_kernel(ListArgs a) {
  __shared__ unsigned char cls[kListChunk];
  __shared__ int wsum[2][kListWarps];
  __shared__ int s_base[2];
  const int nfix = FWD ? a.nqb : a.nkb, nstr = FWD ? a.nkb : a.nqb;
  const int bh = blockIdx.x / nfix, f = blockIdx.x % nfix;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)bh * nfix + f;
  int32_t* midx = (FWD ? a.q_mask_idx : a.k_mask_idx) + row * nstr;
  int32_t* fidx = (FWD ? a.q_full_idx : a.k_full_idx) + row * nstr;
  if (threadIdx.x == 0) s_base[0] = s_base[1] = 0;
  for (int c0 = 0; c0 < nstr; c0 += kListChunk) {
    const int n = min(kListChunk, nstr - c0);
    for (int j = warp; j < n; j += kListWarps) {
      const int sb = c0 + j;
      const int cl = FWD ? block_class(a, bh, f, sb) : block_class(a, bh, sb, f);
      if (lane == 0) cls[j] = (unsigned char)cl;
    }
    __syncthreads();
    const int t = threadIdx.x;
    const int cl = t < n ? cls[t] : 0;
    const unsigned bm = __ballot_sync(0xffffffffu, cl == 1), bf = __ballot_sync(0xffffffffu, cl == 2);
    if (lane == 0) {
      wsum[0][warp] = __popc(bm);
      wsum[1][warp] = __popc(bf);
    }
    __syncthreads();
    int om = s_base[0], of = s_base[1];
    for (int w = 0; w < warp; ++w) {
      om += wsum[0][w];
      of += wsum[1][w];
    }
    const unsigned below = (1u << lane) - 1u;
    if (cl == 1) midx[om + __popc(bm & below)] = c0 + t;
    if (cl == 2) fidx[of + __popc(bf & below)] = c0 + t;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 0; w < kListWarps; ++w) {
        s_base[0] += wsum[0][w];
        s_base[1] += wsum[1][w];
      }
    }
    __syncthreads();
  }
  const int nm = s_base[0], nf = s_base[1];
  for (int t = nm + threadIdx.x; t < nstr; t += blockDim.x) midx[t] = 0;
  for (int t = nf + threadIdx.x; t < nstr; t += blockDim.x) fidx[t] = 0;
  if (threadIdx.x == 0) {
    (FWD ? a.q_mask_cnt : a.k_mask_cnt)[row] = nm;
    (FWD ? a.q_full_cnt : a.k_full_cnt)[row] = nf;
  }
}

int blockmask_launch(int B, int H, int Sq, int Sk, const HostMask& m, const gbattn_blocks* out, cudaStream_t st) {
  ListArgs a;
  memset(&a, 0, sizeof(a));
  a.mask.kind = m.kind;
  a.mask.window_left = m.window_left;
  a.mask.block_size = m.block_size;
  a.mask.prefix_len = m.prefix_len;
  a.mask.nkw = (Sk + 31) / 32;
  a.mask.table = m.kind == GBATTN_MASK_TABLE ? m.table : nullptr;
  a.mask.table_per_head = m.table_per_head;
  a.Sq = Sq;
  a.Sk = Sk;
  a.sm = out->sparse_m;
  a.sn = out->sparse_n;
  a.nqb = (Sq + a.sm - 1) / a.sm;
  a.nkb = (Sk + a.sn - 1) / a.sn;
  a.BH = B * H;
  a.q_mask_cnt = out->q_mask_cnt;
  a.q_mask_idx = out->q_mask_idx;
  a.q_full_cnt = out->q_full_cnt;
  a.q_full_idx = out->q_full_idx;
  a.k_mask_cnt = out->k_mask_cnt;
  a.k_mask_idx = out->k_mask_idx;
  a.k_full_cnt = out->k_full_cnt;
  a.k_full_idx = out->k_full_idx;
  if (m.kind == GBATTN_MASK_DYNAMIC_TOPK) {
    topk_keep_kernel<<<a.BH, kTopkThreads, 0, st>>>(m.key_bias, Sk, m.topk, out->keep_bits, a.mask.nkw);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
    a.mask.keep = out->keep_bits;
    if (out->keep_idx) {
      keep_index_kernel<<<a.BH, kTopkThreads, 0, st>>>(out->keep_bits, Sk, a.mask.nkw, out->keep_idx);
      if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
    }
  }
  const long long cf = (long long)a.BH * a.nqb, cb = (long long)a.BH * a.nkb;
  if (cf >= (1ll << 31) || cb >= (1ll << 31)) return GBATTN_ERR_ARG;
  lists_kernel<true><<<(unsigned)cf, kListWarps * 32, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  lists_kernel<false><<<(unsigned)cb, kListWarps * 32, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;
  return GBATTN_OK;
}

GB_DEFINE_ERROR_READER(blockmask_take_error)

}  // namespace gb
