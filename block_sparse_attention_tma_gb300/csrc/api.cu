// api.cu - the C ABI of libgbattn.so: host-side argument checks, tensor-map
// encoding and dispatch to the kernels. Every check runs before the first
// CUDA call, so a rejected call touches no device state.
#include <math.h>
#include <string.h>

#include <mutex>

#include "kernels.h"
#include "../../include/gbattn_test.h"

namespace gb {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

namespace {
// gbattn_set_dkdv_cta_pair: -1 = library default, 0 = one-CTA kernel, 1 = CTA pair
std::atomic<int> g_dkdv_pair{-1};
constexpr bool kDkdvPairDefault = false;
}  // namespace

bool dkdv_cta_pair_enabled() {
  const int v = g_dkdv_pair.load(std::memory_order_relaxed);
  return v < 0 ? kDkdvPairDefault : v != 0;
}

size_t bwd_workspace_bytes(const Shape& s) {
  const size_t BH = (size_t)s.B * s.H;
  const size_t sq_pad = align_up((size_t)s.Sq, 128);
  return 2 * align_up(BH * sq_pad * sizeof(float), 256);
}

namespace {

constexpr int kMaxSeq = 1 << 30;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool dims_ok(int B, int H, int Sq, int Sk) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return false;
  if (Sq > kMaxSeq || Sk > kMaxSeq) return false;
  const long long bh = (long long)B * H;
  if (bh > (1ll << 24)) return false;
  // one CTA per 128-row tile: keep every grid within 2^31 - 1 blocks
  if (bh * ((Sq + 127) / 128) >= (1ll << 31) || bh * ((Sk + 127) / 128) >= (1ll << 31)) return false;
  return true;
}

// Grouped-query attention: H query heads share Hkv key/value heads.
bool heads_ok(int H, int Hkv) { return Hkv >= 1 && Hkv <= H && H % Hkv == 0; }

// The tensor-core kernels keep 128-row / 128-key tile indices in 15 bits.
bool bf16_seq_ok(int Sq, int Sk) { return (Sq + 127) / 128 < 32768 && (Sk + 127) / 128 < 32768; }

bool bf16_dims_ok(int Dqk, int Dv) {
  return (Dqk == 32 && Dv == 32) || (Dqk == 64 && Dv == 64) || (Dqk == 128 && Dv == 128) ||
         (Dqk == 192 && Dv == 128);
}
bool fp32_dims_ok(int Dqk, int Dv) { return Dqk >= 1 && Dqk <= 128 && Dv >= 1 && Dv <= 128; }

// Device must be compute capability 10.3; cached per device ordinal.
int device_check() {
  static std::mutex mu;
  static int cached[64];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return GBATTN_ERR_UNSUPPORTED;
  }
  if (dev < 64) {
    std::lock_guard<std::mutex> g(mu);
    if (cached[dev] != 0) return cached[dev] > 0 ? GBATTN_OK : GBATTN_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return GBATTN_ERR_UNSUPPORTED;
  }
  const bool ok = (major == 10 && minor == 3);
  if (dev < 64) {
    std::lock_guard<std::mutex> g(mu);
    cached[dev] = ok ? 1 : -1;
  }
  return ok ? GBATTN_OK : GBATTN_ERR_UNSUPPORTED;
}

// Checks the mask struct; fills the scalar part of hm.
int check_mask(const gbattn_mask* mask, HostMask* hm) {
  memset(hm, 0, sizeof(*hm));
  hm->kind = GBATTN_MASK_NONE;
  hm->window_left = -1;
  if (!mask) return GBATTN_OK;
  if (mask->kind < GBATTN_MASK_NONE || mask->kind > GBATTN_MASK_TABLE) return GBATTN_ERR_ARG;
  if (mask->kind == GBATTN_MASK_TABLE && !mask->table) return GBATTN_ERR_ARG;
  if (mask->table && !aligned4(mask->table)) return GBATTN_ERR_ALIGN;
  if ((mask->kind == GBATTN_MASK_BLOCK_DIAG || mask->kind == GBATTN_MASK_MINI_CAUSAL) && mask->block_size <= 0)
    return GBATTN_ERR_ARG;
  if (mask->kind == GBATTN_MASK_PREFIX_LM && mask->prefix_len < 0) return GBATTN_ERR_ARG;
  if (mask->kind == GBATTN_MASK_DYNAMIC_TOPK && (mask->topk < 0 || !mask->key_bias)) return GBATTN_ERR_ARG;
  if (!isfinite(mask->softcap) || mask->softcap < 0.f || !isfinite(mask->rel_bias_slope)) return GBATTN_ERR_ARG;
  if (mask->key_bias && !aligned4(mask->key_bias)) return GBATTN_ERR_ALIGN;
  hm->kind = mask->kind;
  hm->window_left = mask->kind == GBATTN_MASK_SLIDING ? mask->window_left : -1;
  hm->block_size = mask->block_size;
  hm->prefix_len = mask->prefix_len;
  hm->topk = mask->topk;
  hm->slope = mask->rel_bias_slope;
  hm->softcap = mask->softcap;
  hm->key_bias = mask->key_bias;
  hm->table = mask->kind == GBATTN_MASK_TABLE ? mask->table : nullptr;
  hm->table_per_head = mask->table_per_head != 0;
  return GBATTN_OK;
}

int check_tiles(const gbattn_blocks* b) {
  if (b->sparse_m < 128 || b->sparse_n < 128 || (b->sparse_m % 128) || (b->sparse_n % 128)) return GBATTN_ERR_BLOCKS;
  if (b->sparse_m > (1 << 20) || b->sparse_n > (1 << 20)) return GBATTN_ERR_BLOCKS;
  return GBATTN_OK;
}

// Attaches the block lists (forward: need_fwd, backward: need_bwd).
int check_blocks(const gbattn_blocks* b, int Sq, int Sk, bool need_fwd, bool need_bwd, HostMask* hm) {
  if (!b) {
    if (hm->kind != GBATTN_MASK_NONE) return GBATTN_ERR_BLOCKS;
    hm->has_lists = 0;
    return GBATTN_OK;
  }
  int rc = check_tiles(b);
  if (rc) return rc;
  if (need_fwd && (!b->q_mask_cnt || !b->q_mask_idx || !b->q_full_cnt || !b->q_full_idx)) return GBATTN_ERR_BLOCKS;
  if (need_bwd && (!b->k_mask_cnt || !b->k_mask_idx || !b->k_full_cnt || !b->k_full_idx)) return GBATTN_ERR_BLOCKS;
  if (hm->kind == GBATTN_MASK_DYNAMIC_TOPK && !b->keep_bits) return GBATTN_ERR_BLOCKS;
  hm->has_lists = 1;
  hm->sparse_m = b->sparse_m;
  hm->sparse_n = b->sparse_n;
  hm->nqb = (Sq + b->sparse_m - 1) / b->sparse_m;
  hm->nkb = (Sk + b->sparse_n - 1) / b->sparse_n;
  hm->q_mask_cnt = b->q_mask_cnt;
  hm->q_mask_idx = b->q_mask_idx;
  hm->q_full_cnt = b->q_full_cnt;
  hm->q_full_idx = b->q_full_idx;
  hm->k_mask_cnt = b->k_mask_cnt;
  hm->k_mask_idx = b->k_mask_idx;
  hm->k_full_cnt = b->k_full_cnt;
  hm->k_full_idx = b->k_full_idx;
  hm->keep = b->keep_bits;
  hm->keep_idx = b->keep_idx;
  return GBATTN_OK;
}

// Gathered keys: the bf16 kernels stream only the kept keys of a dynamic
// mask when the caller passed the kept-key index list (row indices of the
// 2-D gather maps must fit in int32).
void choose_gather(int dtype, const Shape& s, HostMask* hm) {
  hm->gather = 0;
  hm->kept = s.Sk;
  if (dtype != GBATTN_BF16 || hm->kind != GBATTN_MASK_DYNAMIC_TOPK || !hm->has_lists || !hm->keep_idx) return;
  if (s.Hkv != s.H) return;  // compact key tiles are per query head
  if ((long long)s.B * s.H * s.Sk >= (1ll << 31)) return;
  hm->gather = 1;
  hm->kept = hm->topk < s.Sk ? hm->topk : s.Sk;
}

float resolve_scale(float scale, int Dqk) { return (scale > 0.f && isfinite(scale)) ? scale : 1.0f / sqrtf((float)Dqk); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, int S, int BH, int swizzle_bytes) {
  return make_tmap_bf16_3d_box(map, base, D, S, BH, swizzle_bytes, 128);
}

bool make_tmap_bf16_3d_box(CUtensorMap* map, const void* base, int D, int S, int BH, int swizzle_bytes,
                           int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)(swizzle_bytes / 2), (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_rows(CUtensorMap* map, const void* base, int D, long long rows, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {(cuuint32_t)(swizzle_bytes / 2), 1};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace gb

using namespace gb;

extern "C" {

int gbattn_version(void) { return 102; }

const char* gbattn_strerror(int status) {
  switch (status) {
    case GBATTN_OK: return "ok";
    case GBATTN_ERR_ARG: return "invalid argument (null pointer or bad dimension)";
    case GBATTN_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case GBATTN_ERR_UNSUPPORTED: return "unsupported dtype/head-dim combination or device is not compute capability 10.3";
    case GBATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case GBATTN_ERR_BLOCKS: return "block-sparse lists missing or inconsistent with the shape";
    case GBATTN_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case GBATTN_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

int gbattn_block_mask_sizes(int B, int H, int Sq, int Sk, int sparse_m, int sparse_n, size_t* q_cnt_bytes,
                            size_t* q_idx_bytes, size_t* k_cnt_bytes, size_t* k_idx_bytes,
                            size_t* keep_bits_bytes, size_t* keep_idx_bytes) {
  if (!dims_ok(B, H, Sq, Sk)) return GBATTN_ERR_ARG;
  if (sparse_m < 128 || sparse_n < 128 || sparse_m % 128 || sparse_n % 128) return GBATTN_ERR_ARG;
  const size_t BH = (size_t)B * H;
  const size_t nqb = (Sq + sparse_m - 1) / sparse_m, nkb = (Sk + sparse_n - 1) / sparse_n;
  if (q_cnt_bytes) *q_cnt_bytes = BH * nqb * 4;
  if (q_idx_bytes) *q_idx_bytes = BH * nqb * nkb * 4;
  if (k_cnt_bytes) *k_cnt_bytes = BH * nkb * 4;
  if (k_idx_bytes) *k_idx_bytes = BH * nkb * nqb * 4;
  if (keep_bits_bytes) *keep_bits_bytes = BH * ((Sk + 31) / 32) * 4;
  if (keep_idx_bytes) *keep_idx_bytes = BH * (size_t)Sk * 4;
  return GBATTN_OK;
}

int build_block_mask(int B, int H, int Sq, int Sk, const gbattn_mask* mask, gbattn_blocks* out,
                     gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || !out) return GBATTN_ERR_ARG;
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  rc = check_tiles(out);
  if (rc) return rc;
  if (!out->q_mask_cnt || !out->q_mask_idx || !out->q_full_cnt || !out->q_full_idx || !out->k_mask_cnt ||
      !out->k_mask_idx || !out->k_full_cnt || !out->k_full_idx)
    return GBATTN_ERR_ARG;
  if (hm.kind == GBATTN_MASK_DYNAMIC_TOPK && !out->keep_bits) return GBATTN_ERR_ARG;
  if (out->keep_idx && !aligned4(out->keep_idx)) return GBATTN_ERR_ALIGN;
  rc = device_check();
  if (rc) return rc;
  return blockmask_launch(B, H, Sq, Sk, hm, out, static_cast<cudaStream_t>(stream));
}

int attn_fwd(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv, const void* q, const void* k,
             const void* v, float scale, const gbattn_mask* mask, const gbattn_blocks* blocks, void* o, float* lse,
             gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || Dqk < 1 || Dv < 1 || !heads_ok(H, Hkv)) return GBATTN_ERR_ARG;
  if (!q || !k || !v || !o) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned4(lse)))
    return GBATTN_ERR_ALIGN;
  if (dtype == GBATTN_BF16) {
    if (!bf16_dims_ok(Dqk, Dv) || !bf16_seq_ok(Sq, Sk)) return GBATTN_ERR_UNSUPPORTED;
  } else if (dtype == GBATTN_FP32) {
    if (!fp32_dims_ok(Dqk, Dv)) return GBATTN_ERR_UNSUPPORTED;
  } else {
    return GBATTN_ERR_UNSUPPORTED;
  }
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  rc = check_blocks(blocks, Sq, Sk, true, false, &hm);
  if (rc) return rc;
  rc = device_check();
  if (rc) return rc;
  const Shape s{B, H, Sq, Sk, Dqk, Dv, Hkv};
  choose_gather(dtype, s, &hm);
  const float sc = resolve_scale(scale, Dqk);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GBATTN_BF16) return fwd_bf16_launch(s, q, k, v, sc, hm, o, lse, st);
  return fwd_fp32_launch(s, static_cast<const float*>(q), static_cast<const float*>(k),
                         static_cast<const float*>(v), sc, hm, static_cast<float*>(o), lse, st);
}

size_t attn_bwd_workspace_bytes(int dtype, int B, int H, int Sq, int Sk, int Dqk, int Dv) {
  if (!dims_ok(B, H, Sq, Sk) || Dqk < 1 || Dv < 1) return 0;
  if (dtype != GBATTN_BF16 && dtype != GBATTN_FP32) return 0;
  return bwd_workspace_bytes(Shape{B, H, Sq, Sk, Dqk, Dv, H});
}

int attn_bwd(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv, const void* q, const void* k,
             const void* v, const void* o, const void* dout, const float* lse, float scale, const gbattn_mask* mask,
             const gbattn_blocks* blocks, int deterministic, void* dq, void* dk, void* dv, float* dkey_bias,
             void* workspace, size_t workspace_bytes, gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || Dqk < 1 || Dv < 1 || !heads_ok(H, Hkv)) return GBATTN_ERR_ARG;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return GBATTN_ERR_ARG;
  if (deterministic != 0 && deterministic != 1) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (dkey_bias && !aligned4(dkey_bias)))
    return GBATTN_ERR_ALIGN;
  if (dtype == GBATTN_BF16) {
    if (!bf16_dims_ok(Dqk, Dv) || !bf16_seq_ok(Sq, Sk)) return GBATTN_ERR_UNSUPPORTED;
  } else if (dtype == GBATTN_FP32) {
    if (!fp32_dims_ok(Dqk, Dv)) return GBATTN_ERR_UNSUPPORTED;
  } else {
    return GBATTN_ERR_UNSUPPORTED;
  }
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  rc = check_blocks(blocks, Sq, Sk, true, true, &hm);
  if (rc) return rc;
  const Shape s{B, H, Sq, Sk, Dqk, Dv, Hkv};
  if (Hkv != H) {
    // the key-bias gradient is per query head; a group's dK/dV kernel walks
    // G heads' tiles under one 15-bit tile index
    if (dkey_bias) return GBATTN_ERR_UNSUPPORTED;
    if (H / Hkv > kMaxGroup || (long long)(H / Hkv) * ((Sq + 127) / 128) >= 32768) return GBATTN_ERR_UNSUPPORTED;
  }
  if (!workspace || workspace_bytes < bwd_workspace_bytes(s)) return GBATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GBATTN_ERR_ALIGN;
  rc = device_check();
  if (rc) return rc;
  choose_gather(dtype, s, &hm);
  const float sc = resolve_scale(scale, Dqk);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GBATTN_BF16)
    return bwd_bf16_launch(s, q, k, v, o, dout, lse, sc, hm, dq, dk, dv, dkey_bias, workspace, st);
  return bwd_fp32_launch(s, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
                         static_cast<const float*>(o), static_cast<const float*>(dout), lse, sc, hm,
                         static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv), dkey_bias,
                         workspace, st);
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Sq, int Dv, int num_splits) {
  if (B < 1 || H < 1 || Sq < 1 || Dv < 1 || num_splits < 1 || num_splits > 64) return 0;
  if (num_splits == 1) return 0;
  const size_t rows = (size_t)num_splits * B * H * Sq;
  return align_up(rows * Dv * sizeof(float), 256) + align_up(rows * sizeof(float), 256);
}

int attn_fwd_splitkv(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv, const void* q,
                     const void* k, const void* v, float scale, const gbattn_mask* mask, int num_splits, void* o,
                     float* lse, void* workspace, size_t workspace_bytes, gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || Dqk < 1 || Dv < 1 || !heads_ok(H, Hkv)) return GBATTN_ERR_ARG;
  if (!q || !k || !v || !o) return GBATTN_ERR_ARG;
  if (num_splits < 1 || num_splits > 64) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned4(lse)))
    return GBATTN_ERR_ALIGN;
  if (dtype != GBATTN_BF16) return GBATTN_ERR_UNSUPPORTED;
  if (!(Dqk == Dv && (Dqk == 64 || Dqk == 128))) return GBATTN_ERR_UNSUPPORTED;
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  if (hm.kind != GBATTN_MASK_NONE && hm.kind != GBATTN_MASK_CAUSAL) return GBATTN_ERR_UNSUPPORTED;
  if (hm.softcap != 0.f || hm.slope != 0.f || hm.key_bias) return GBATTN_ERR_UNSUPPORTED;
  if (num_splits > 1) {
    if (!workspace || workspace_bytes < attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits))
      return GBATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GBATTN_ERR_ALIGN;
  }
  rc = device_check();
  if (rc) return rc;
  const Shape s{B, H, Sq, Sk, Dqk, Dv, Hkv};
  return splitkv_launch(s, q, k, v, resolve_scale(scale, Dqk), hm.kind == GBATTN_MASK_CAUSAL, num_splits, o, lse,
                        workspace, static_cast<cudaStream_t>(stream), nullptr);
}

int attn_fwd_splitkv_paged(int dtype, int B, int H, int Hkv, int Sq, int Dqk, int Dv, const void* q,
                           const void* k_cache, const void* v_cache, int num_pages, int page_size,
                           const int32_t* page_table, int max_pages_per_seq, const int32_t* seqlens_k, float scale,
                           const gbattn_mask* mask, int num_splits, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, gbattn_stream stream) {
  if (B < 1 || H < 1 || Sq < 1 || Dqk < 1 || Dv < 1 || !heads_ok(H, Hkv)) return GBATTN_ERR_ARG;
  if ((long long)B * H > (1ll << 24) || Sq > kMaxSeq) return GBATTN_ERR_ARG;
  if (!q || !k_cache || !v_cache || !o || !page_table || !seqlens_k) return GBATTN_ERR_ARG;
  if (num_pages < 1 || page_size < 64 || page_size % 64 || max_pages_per_seq < 1) return GBATTN_ERR_ARG;
  if ((long long)max_pages_per_seq * page_size > kMaxSeq) return GBATTN_ERR_ARG;
  if ((long long)num_pages * Hkv * page_size >= (1ll << 31)) return GBATTN_ERR_ARG;
  if (num_splits < 1 || num_splits > 64) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || (lse && !aligned4(lse)) ||
      !aligned4(page_table) || !aligned4(seqlens_k))
    return GBATTN_ERR_ALIGN;
  if (dtype != GBATTN_BF16) return GBATTN_ERR_UNSUPPORTED;
  if (!(Dqk == Dv && (Dqk == 64 || Dqk == 128))) return GBATTN_ERR_UNSUPPORTED;
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  if (hm.kind != GBATTN_MASK_NONE && hm.kind != GBATTN_MASK_CAUSAL) return GBATTN_ERR_UNSUPPORTED;
  if (hm.softcap != 0.f || hm.slope != 0.f || hm.key_bias) return GBATTN_ERR_UNSUPPORTED;
  if (num_splits > 1) {
    if (!workspace || workspace_bytes < attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits))
      return GBATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GBATTN_ERR_ALIGN;
  }
  rc = device_check();
  if (rc) return rc;
  const Shape s{B, H, Sq, max_pages_per_seq * page_size, Dqk, Dv, Hkv};
  const PagedKV pk{seqlens_k, page_table, page_size, max_pages_per_seq, num_pages};
  return splitkv_launch(s, q, k_cache, v_cache, resolve_scale(scale, Dqk), hm.kind == GBATTN_MASK_CAUSAL,
                        num_splits, o, lse, workspace, static_cast<cudaStream_t>(stream), &pk);
}

int attn_fwd_splitkv_noalloc(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv, const void* q,
                             const void* k, const void* v, float scale, const gbattn_mask* mask, int num_splits,
                             void* o, float* lse, gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || Dqk < 1 || Dv < 1 || !heads_ok(H, Hkv)) return GBATTN_ERR_ARG;
  if (!q || !k || !v || !o) return GBATTN_ERR_ARG;
  if (num_splits < 1 || num_splits > 64) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned4(lse)))
    return GBATTN_ERR_ALIGN;
  if (dtype != GBATTN_BF16) return GBATTN_ERR_UNSUPPORTED;
  if (!(Dqk == Dv && (Dqk == 64 || Dqk == 128))) return GBATTN_ERR_UNSUPPORTED;
  HostMask hm;
  int rc = check_mask(mask, &hm);
  if (rc) return rc;
  if (hm.kind != GBATTN_MASK_NONE && hm.kind != GBATTN_MASK_CAUSAL) return GBATTN_ERR_UNSUPPORTED;
  if (hm.softcap != 0.f || hm.slope != 0.f || hm.key_bias) return GBATTN_ERR_UNSUPPORTED;
  const size_t need = attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits);
  if (need > (size_t)GBATTN_NOALLOC_SCRATCH_BYTES) return GBATTN_ERR_WORKSPACE;
  rc = device_check();
  if (rc) return rc;
  const Shape s{B, H, Sq, Sk, Dqk, Dv, Hkv};
  return splitkv_noalloc_launch(s, q, k, v, resolve_scale(scale, Dqk), hm.kind == GBATTN_MASK_CAUSAL, num_splits,
                                need, o, lse, static_cast<cudaStream_t>(stream));
}

int gbattn_test_fwd_stalled(int B, int H, int Sq, int Sk, int D, const void* q, const void* k, const void* v,
                            void* o, float* lse, unsigned long long wait_ns, gbattn_stream stream) {
  if (!dims_ok(B, H, Sq, Sk) || !q || !k || !v || !o || !lse) return GBATTN_ERR_ARG;
  if (wait_ns < 1 || wait_ns > 2000000000ull) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse)) return GBATTN_ERR_ALIGN;
  if (D != 32 && D != 64 && D != 128) return GBATTN_ERR_UNSUPPORTED;
  if (!bf16_seq_ok(Sq, Sk)) return GBATTN_ERR_UNSUPPORTED;
  const int rc = device_check();
  if (rc) return rc;
  HostMask hm;
  check_mask(nullptr, &hm);
  const Shape s{B, H, Sq, Sk, D, D, H};
  const FwdTestHook hook{wait_ns, 1};
  return fwd_bf16_launch(s, q, k, v, resolve_scale(0.f, D), hm, o, lse, static_cast<cudaStream_t>(stream), &hook);
}

int gbattn_test_bwd_stalled(int B, int H, int S, int D, const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, unsigned long long wait_ns, gbattn_stream stream) {
  if (!dims_ok(B, H, S, S) || !q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return GBATTN_ERR_ARG;
  if (wait_ns < 1 || wait_ns > 2000000000ull) return GBATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return GBATTN_ERR_ALIGN;
  if (D != 32 && D != 64 && D != 128) return GBATTN_ERR_UNSUPPORTED;
  if (!bf16_seq_ok(S, S)) return GBATTN_ERR_UNSUPPORTED;
  const Shape s{B, H, S, S, D, D, H};
  if (!workspace || workspace_bytes < bwd_workspace_bytes(s)) return GBATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GBATTN_ERR_ALIGN;
  const int rc = device_check();
  if (rc) return rc;
  HostMask hm;
  check_mask(nullptr, &hm);
  const BwdTestHook hook{wait_ns, 1};
  return bwd_bf16_launch(s, q, k, v, o, dout, lse, resolve_scale(0.f, D), hm, dq, dk, dv, nullptr, workspace,
                         static_cast<cudaStream_t>(stream), &hook);
}

int gbattn_set_dkdv_cta_pair(int mode, int* previous) {
  if (mode < -1 || mode > 1) return GBATTN_ERR_ARG;
  const int prev = g_dkdv_pair.exchange(mode);
  if (previous) *previous = prev;
  return GBATTN_OK;
}

int gbattn_last_device_error(gbattn_stream stream) {
  if (device_check() != GBATTN_OK) return GBATTN_ERR_UNSUPPORTED;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GBATTN_ERR_CUDA;
  int errs[7] = {fwd_take_error(),    bwd_take_error(),    dkdv_take_error(),   dkdv2_take_error(),
                 simt_take_error(),   decode_take_error(), blockmask_take_error()};
  for (int e : errs)
    if (e == GBATTN_ERR_CUDA) return e;
  for (int e : errs)
    if (e == GBATTN_ERR_TIMEOUT) return e;
  for (int e : errs)
    if (e != 0) return e;
  return GBATTN_OK;
}

}  // extern "C"
