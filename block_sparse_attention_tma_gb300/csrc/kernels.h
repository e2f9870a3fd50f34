// kernels.h - host-side interface between the C ABI (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/gbattn.h"

namespace gb {

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device. The attribute belongs to the function in one device's context, so
// it is set once per device ordinal: `done` holds one bit per device (< 64;
// higher ordinals set it on every launch). Two host threads may both set it
// the first time, which is harmless.
template <typename K>
inline int ensure_smem(K kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GBATTN_ERR_CUDA;
  }
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return GBATTN_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return GBATTN_ERR_CUDA;
  }
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return GBATTN_OK;
}

// L2 size of the current device in bytes (cached per device ordinal; 128 MB
// if the query fails).
inline long long device_l2_bytes() {
  static std::atomic<long long> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 128ll << 20;
  }
  if (dev >= 0 && dev < 64) {
    const long long c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int l2 = 0;
  long long v = 128ll << 20;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) == cudaSuccess && l2 > 0) v = l2;
  else cudaGetLastError();
  if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// CTA order of the prefill kernels: heads are taken in groups of this many,
// each group's tiles in the kernel's own (heaviest-first) order, so that the
// tiles in flight stream the operands of a few heads only and those stay in
// L2. 0 (no grouping) when every head's streamed bytes fit in half the L2
// anyway; otherwise as many heads as fit in 3/8 of it (at least 1).
inline int head_group(long long heads, long long bytes_per_head, long long l2_bytes) {
  if (heads <= 1 || bytes_per_head <= 0 || heads * bytes_per_head <= l2_bytes / 2) return 0;
  const long long g = (l2_bytes * 3 / 8) / bytes_per_head;
  return (int)(g < 1 ? 1 : (g >= heads ? 0 : g));
}

// Tile of block b in a grid of `heads` x `ntiles` CTAs: head h and tile
// index t (0 = the first tile in the kernel's order), with heads grouped by
// `grp` (0: tile-major over all heads, head = b % heads).
__host__ __device__ inline void grid_tile(int b, int heads, int ntiles, int grp, int* h, int* t) {
  if (grp <= 0) {
    *h = b % heads;
    *t = b / heads;
    return;
  }
  const int ngr = (heads + grp - 1) / grp;
  int g = b / (grp * ntiles);
  if (g > ngr - 1) g = ngr - 1;
  const int r = b - g * grp * ntiles;
  const int gs = heads - g * grp < grp ? heads - g * grp : grp;
  *h = g * grp + r % gs;
  *t = r / gs;
}

// Largest number of query heads per key/value head (GQA group) the
// tensor-core backward accepts.
constexpr int kMaxGroup = 128;

struct Shape {
  int B, H, Sq, Sk, Dqk, Dv;
  int Hkv;  // key/value heads (H % Hkv == 0; Hkv == H without GQA)
};

// Validated, device-ready view of the mask and lists of one call.
struct HostMask {
  int kind, window_left, block_size, prefix_len, topk;
  float slope, softcap;
  const float* key_bias;
  const uint32_t* keep;
  const uint32_t* table;  // element table (mask kind TABLE)
  int table_per_head;
  int has_lists;
  int sparse_m, sparse_n, nqb, nkb;
  const int32_t *q_mask_cnt, *q_mask_idx, *q_full_cnt, *q_full_idx;
  const int32_t *k_mask_cnt, *k_mask_idx, *k_full_cnt, *k_full_idx;
  // gathered keys (bf16 DYNAMIC_TOPK with the kept-key index list): the
  // kernels stream only the `kept` = min(topk, Sk) keys listed in keep_idx
  int gather, kept;
  const int32_t* keep_idx;
};

// Encodes a 3-D bf16 tensor map over [BH, S, D] (D innermost) with a box of
// (swizzle_bytes/2) x 128 x 1 and the given swizzle (64 or 128 bytes).
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, int S, int BH, int swizzle_bytes);
// The same with a box of (swizzle_bytes/2) x box_rows x 1.
bool make_tmap_bf16_3d_box(CUtensorMap* map, const void* base, int D, int S, int BH, int swizzle_bytes,
                           int box_rows);
// Encodes a 2-D bf16 tensor map over [rows, D] with a box one row high and
// (swizzle_bytes/2) wide, for TMA row gathers (tile::gather4).
bool make_tmap_bf16_rows(CUtensorMap* map, const void* base, int D, long long rows, int swizzle_bytes);

// Test hook of the bf16 forward (the abort path of its bounded waits): a
// shorter wait limit, and the K tile of the first visited tile withheld so
// that the MMA thread's wait for it runs out.
struct FwdTestHook {
  unsigned long long wait_ns;
  int withhold_first_k_tile;
};

// Kernel launchers: return GBATTN_OK or GBATTN_ERR_CUDA.
int fwd_bf16_launch(const Shape& s, const void* q, const void* k, const void* v, float scale,
                    const HostMask& m, void* o, float* lse, cudaStream_t st, const FwdTestHook* hook = nullptr);
int fwd_fp32_launch(const Shape& s, const float* q, const float* k, const float* v, float scale,
                    const HostMask& m, float* o, float* lse, cudaStream_t st);
// Test hook of the bf16 backward: a shorter wait limit, and the dO tile of
// each dK/dV CTA's first query tile and the K tile of each dQ CTA's first key
// tile withheld, so that the MMA issuers' waits for them run out.
struct BwdTestHook {
  unsigned long long wait_ns;
  int withhold_first_tiles;
};
int bwd_bf16_launch(const Shape& s, const void* q, const void* k, const void* v, const void* o,
                    const void* dout, const float* lse, float scale, const HostMask& m, void* dq, void* dk,
                    void* dv, float* dkey_bias, void* ws, cudaStream_t st, const BwdTestHook* hook = nullptr);
int bwd_fp32_launch(const Shape& s, const float* q, const float* k, const float* v, const float* o,
                    const float* dout, const float* lse, float scale, const HostMask& m, float* dq, float* dk,
                    float* dv, float* dkey_bias, void* ws, cudaStream_t st);
// Paged key/value cache of the decode path: pages of page_size keys of one
// key/value head ([num_pages, Hkv, page_size, D]); seqlens may be given
// without a page table (a dense cache with per-sequence key counts).
struct PagedKV {
  const int32_t* seqlens;     // [B] or nullptr
  const int32_t* page_table;  // [B][max_pages] or nullptr
  int page_size, max_pages, num_pages;
};
// Split-KV decode of grouped query heads on the tensor cores (the forward
// kernel in packed mode): writes O / LSE directly (num_splits == 1) or the
// split partials o_part / lse_part for the combine. D = 64 / 128; a dense
// cache, or a paged one whose pages hold a multiple of 128 keys.
int fwd_packed_decode_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                             int num_splits, void* o, float* lse, float* o_part, float* lse_part,
                             const PagedKV* paged, cudaStream_t st);
int splitkv_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                   int num_splits, void* o, float* lse, void* ws, cudaStream_t st, const PagedKV* paged);
// Split-KV forward with its split partials in the library's static scratch
// array (no allocation); workspace_bytes is what attn_fwd_splitkv would need.
int splitkv_noalloc_launch(const Shape& s, const void* q, const void* k, const void* v, float scale, int causal,
                           int num_splits, size_t workspace_bytes, void* o, float* lse, cudaStream_t st);
int blockmask_launch(int B, int H, int Sq, int Sk, const HostMask& m, const gbattn_blocks* out,
                     cudaStream_t st);

// Device error words, one per translation unit (read and cleared).
int fwd_take_error();
int bwd_take_error();
int dkdv_take_error();
int dkdv2_take_error();
int simt_take_error();
int decode_take_error();
int blockmask_take_error();

// Which dK/dV kernel attn_bwd runs where the CTA-pair kernel applies
// (gbattn_set_dkdv_cta_pair; process-wide).
bool dkdv_cta_pair_enabled();

// Workspace layout of attn_bwd: [delta fp32 BH x ceil128(Sq)][lse2 fp32 BH x ceil128(Sq)]
size_t bwd_workspace_bytes(const Shape& s);
size_t align_up(size_t x, size_t a);

}  // namespace gb
