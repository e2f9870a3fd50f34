/*
 * gbattn.h - C ABI of libgbattn.so: fused, block-sparse scaled-dot-product
 * attention for one GB300 GPU (compute capability 10.3, sm_103a).
 *
 * What the operations compute is taken from these pages:
 *   [FSA]  "Optimize Flash Dynamic Mask Attention Kernel Configurations"
 *          (flash-sparse-attention PR #148): forward, split-KV forward,
 *          backward with an optional deterministic path; masks and softcap.
 *   [FA2C] "Enable 2CTA for SM100 block-sparse backward" (flash-attention
 *          PR #2661): block-sparse forward/backward driven by per-block index
 *          lists, sparse tiles that are multiples of the kernel tile (q and kv
 *          sub-tiling), mask kinds, QK/V head dims 192/128, rel-bias score_mod.
 *   [PCB]  POPCORNBENCH trace "Kimi-K2.6 l1_p97": scaled-dot-product
 *          attention and the online-softmax merge of partial results.
 *
 * Conventions shared by every entry point
 *   - Layout: Q [B,H,Sq,Dqk], K [B,Hkv,Sk,Dqk], V [B,Hkv,Sk,Dv], O/dO
 *     [B,H,Sq,Dv], each contiguous with the head dim innermost; LSE [B,H,Sq]
 *     fp32. Grouped-query attention ([FA2C]'s reference runs flex_attention
 *     with enable_gqa and the kernel call carries pack_gqa): query head h
 *     reads key/value head h / (H / Hkv); H % Hkv == 0; Hkv == H is plain
 *     multi-head attention. Masks, key biases and block lists are per query
 *     head.
 *   - Every pointer is a DEVICE pointer of the current CUDA device, owned by
 *     the caller. The library allocates nothing, frees nothing and keeps no
 *     pointer after the call returns. Tensor pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Inputs must stay valid until the stream reaches the
 *     end of the work.
 *   - Return value: GBATTN_OK (0) or a negative GBATTN_ERR_* code. Argument
 *     checks run on the host before any CUDA call; nothing is launched when a
 *     check fails. No C++ exception crosses the ABI.
 *   - Mask alignment for Sq != Sk is bottom-right: query i is aligned with key
 *     i + (Sk - Sq).
 *   - Rows with no allowed key produce O = 0, LSE = -inf and zero gradients.
 *   - scale <= 0 selects 1/sqrt(Dqk), the pages' default softmax scale.
 *   - Supported head dims: bf16 (Dqk,Dv) in {(32,32),(64,64),(128,128),
 *     (192,128)} on the tensor-core path; fp32 any 1 <= Dqk,Dv <= 128 on the
 *     exact CUDA-core path. Any Sq, Sk >= 1 (bf16 attn_fwd / attn_bwd: below
 *     2^22, i.e. fewer than 32768 tiles of 128); ragged tile edges are masked.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* gbattn_stream; /* a cudaStream_t */

/* element types */
enum { GBATTN_BF16 = 0, GBATTN_FP32 = 1 };

/* mask kinds ([FA2C] fuzz tester mask names; [FSA] dynamic mask) */
enum {
  GBATTN_MASK_NONE = 0,
  GBATTN_MASK_CAUSAL = 1,       /* key j allowed iff j <= i + (Sk - Sq)                      */
  GBATTN_MASK_SLIDING = 2,      /* 0 <= (i + Sk - Sq) - j <= window_left (window_left < 0:   */
                                /* unbounded, i.e. causal)                                    */
  GBATTN_MASK_BLOCK_DIAG = 3,   /* floor((i + Sk - Sq) / block_size) == floor(j / block_size) */
  GBATTN_MASK_PREFIX_LM = 4,    /* j < prefix_len, or causal                                  */
  GBATTN_MASK_DYNAMIC_TOPK = 5, /* j among the topk keys of (b,h) ranked by key_bias          */
                                /* (descending, ties: lower index first), and causal          */
  GBATTN_MASK_MINI_CAUSAL = 6,  /* causal inside blocks: j <= i + (Sk - Sq) and               */
                                /* floor((i + Sk - Sq) / block_size) == floor(j / block_size) */
                                /* ([FA2C] names mini_causal without defining it; this is the */
                                /* reading taken)                                              */
  GBATTN_MASK_TABLE = 7         /* any element predicate: pair (i, j) allowed iff bit j % 32   */
                                /* of word j / 32 of row i of `table` is set (the caller      */
                                /* evaluates its predicate, e.g. a flex_attention mask_mod,   */
                                /* into the table once; [FA2C] builds block lists from such a */
                                /* predicate)                                                  */
};

/* status codes */
enum {
  GBATTN_OK = 0,
  GBATTN_ERR_ARG = -1,         /* null pointer, non-positive or too large dimension     */
  GBATTN_ERR_ALIGN = -2,       /* a tensor pointer is not 16-byte aligned               */
  GBATTN_ERR_UNSUPPORTED = -3, /* dtype / head-dim combination, or device is not CC 10.3 */
  GBATTN_ERR_WORKSPACE = -4,   /* workspace missing or smaller than the query function says */
  GBATTN_ERR_BLOCKS = -5,      /* block lists missing, or inconsistent with the shape    */
  GBATTN_ERR_CUDA = -6,        /* a CUDA runtime call or a kernel launch failed          */
  GBATTN_ERR_TIMEOUT = -7      /* a kernel gave up a bounded wait (see last_device_error) */
};

/*
 * Element-level mask and score modifiers, shared by every call.
 * Score of pair (i,j): s = scale * q_i.k_j; if softcap > 0, s = softcap *
 * tanh(s / softcap); then s += rel_bias_slope * (i - j) + key_bias[b,h,j].
 * The rel-bias is a constant: the rel-bias score_mod backward of [FA2C]
 * returns the incoming gradient unchanged and nothing flows to the slope.
 * attn_bwd can return the gradient of the key bias on request (dkey_bias).
 */
typedef struct {
  int kind;             /* GBATTN_MASK_*                                        */
  int window_left;      /* SLIDING                                               */
  int block_size;       /* BLOCK_DIAG and MINI_CAUSAL, > 0                       */
  int prefix_len;       /* PREFIX_LM, >= 0                                       */
  int topk;             /* DYNAMIC_TOPK, >= 0                                    */
  float rel_bias_slope; /* 0 = off                                               */
  float softcap;        /* 0 = off                                               */
  const float* key_bias;/* device [B,H,Sk] fp32 additive key bias, or NULL; required */
                        /* for DYNAMIC_TOPK (it is also the ranking key)          */
  const uint32_t* table;/* TABLE: device bits, ceil(Sk/32) uint32 words per query row: */
                        /* [Sq, ceil(Sk/32)] shared by every (b,h), or             */
                        /* [B,H,Sq, ceil(Sk/32)] when table_per_head; bits past Sk */
                        /* are ignored. NULL for the other kinds.                  */
  int table_per_head;   /* 0: one table for all heads; 1: one per (b,h)           */
} gbattn_mask;

/*
 * Block-sparse lists ([FA2C]: forward lists per q-block of kv-blocks, backward
 * lists per kv-block of q-blocks, split into blocks that need the element mask
 * ("mask" lists) and blocks whose every pair is allowed ("full" lists); blocks
 * with no allowed pair are absent and never loaded). Sparse blocks are
 * sparse_m x sparse_n with both multiples of the 128 x 128 kernel tile; the
 * kernels walk each listed block as (sparse_m/128) x (sparse_n/128) tiles.
 * nQB = ceil(Sq/sparse_m), nKB = ceil(Sk/sparse_n). Lists ascend; unused tail
 * entries are 0; a block cut by the end of the sequence is never "full".
 * All arrays are caller-owned device memory (sizes: gbattn_block_mask_sizes).
 */
typedef struct {
  int sparse_m, sparse_n;
  int32_t* q_mask_cnt;  /* [B,H,nQB]     */
  int32_t* q_mask_idx;  /* [B,H,nQB,nKB] */
  int32_t* q_full_cnt;  /* [B,H,nQB]     */
  int32_t* q_full_idx;  /* [B,H,nQB,nKB] */
  int32_t* k_mask_cnt;  /* [B,H,nKB]     */
  int32_t* k_mask_idx;  /* [B,H,nKB,nQB] */
  int32_t* k_full_cnt;  /* [B,H,nKB]     */
  int32_t* k_full_idx;  /* [B,H,nKB,nQB] */
  uint32_t* keep_bits;  /* [B,H,ceil(Sk/32)]: DYNAMIC_TOPK keep set, bit j%32 of word
                           j/32; written by build_block_mask, read by the kernels.
                           NULL allowed for the other kinds.                      */
  int32_t* keep_idx;    /* [B,H,Sk] or NULL: DYNAMIC_TOPK kept-key index list, the
                           min(topk,Sk) kept key indices of each (b,h) ascending,
                           then 0 up to Sk; written by build_block_mask when not
                           NULL. With it, the bf16 attn_fwd / attn_bwd gather only
                           the kept keys into compact 128-key tiles (TMA row
                           gathers) instead of walking the lists with the keep
                           bits; the results are the same. Ignored for the other
                           kinds and by the fp32 path.                             */
} gbattn_blocks;

/* Byte sizes of the block-list arrays for this shape (any of the out pointers
 * may be NULL). Returns GBATTN_ERR_ARG for bad dims or tiles. */
int gbattn_block_mask_sizes(int B, int H, int Sq, int Sk, int sparse_m, int sparse_n,
                            size_t* q_cnt_bytes, size_t* q_idx_bytes,
                            size_t* k_cnt_bytes, size_t* k_idx_bytes,
                            size_t* keep_bits_bytes, size_t* keep_idx_bytes);

/*
 * build_block_mask - classify every sparse block as absent / mask / full and
 * write the forward and backward lists into `out` ([FA2C]
 * `_build_block_sparse_masks_for_bwd`, restated for C). For DYNAMIC_TOPK it
 * first selects the keep set per (b,h) on the GPU and writes out->keep_bits
 * (and out->keep_idx when it is not NULL). The result is exact (integer work;
 * the top-k compares fp32 biases).
 */
int build_block_mask(int B, int H, int Sq, int Sk, const gbattn_mask* mask,
                     gbattn_blocks* out, gbattn_stream stream);

/*
 * attn_fwd - O = softmax(mask(scores)) V and LSE = ln sum_j exp(s_ij), fused:
 * per 128-row query tile the kernel streams the 128-key tiles of the listed
 * blocks, keeps a running max/sum (online softmax, [PCB]) and never writes the
 * score matrix to memory ([FSA] forward; [FA2C] `_flash_attn_fwd` with
 * block_sparse_tensors and return_lse). `blocks` may be NULL only for
 * GBATTN_MASK_NONE. o has the dtype of q; lse may be NULL.
 */
int attn_fwd(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv,
             const void* q, const void* k, const void* v, float scale,
             const gbattn_mask* mask, const gbattn_blocks* blocks,
             void* o, float* lse, gbattn_stream stream);

/* Workspace bytes attn_bwd needs for this shape: two per-row fp32 vectors
 * (rowsum(dO o O) and the log2-domain LSE) of B*H*ceil(Sq/128)*128 entries.
 * Returns 0 for invalid dims. */
size_t attn_bwd_workspace_bytes(int dtype, int B, int H, int Sq, int Sk, int Dqk, int Dv);

/*
 * attn_bwd - gradients of O for the loss <dO, O> ([FSA] backward, "seq-k
 * parallel" path with an optional deterministic mode; [FA2C] `_flash_attn_bwd`
 * with the backward block lists). Steps: D_i = sum_d dO_id O_id; per kv tile
 * (key-parallel), recompute P from LSE, dV += P^T dO, dP = dO V^T,
 * dS = P (dP - D), dK += scale dS^T Q; per query tile (query-parallel),
 * recompute S and dP and accumulate dQ = scale dS K. No gradient is
 * accumulated with atomics, so every output is bitwise reproducible whatever
 * `deterministic` says (0 or 1 are both accepted; any other value is
 * GBATTN_ERR_ARG). o and lse must be the outputs of attn_fwd for the same
 * inputs. workspace is device memory of at least attn_bwd_workspace_bytes();
 * its contents on entry do not matter. With GQA (Hkv < H), dk / dv are
 * [B,Hkv,Sk,D] and sum the contributions of the H / Hkv query heads of each
 * group (one CTA walks all of them, still without atomics); bf16 accepts
 * groups of up to 128 heads with (H/Hkv) * ceil(Sq/128) < 32768, and
 * dkey_bias is not supported with GQA (GBATTN_ERR_UNSUPPORTED).
 * dkey_bias: NULL, or device [B,H,Sk] fp32 (4-byte aligned) that receives the
 * gradient of the loss with respect to key_bias: dkey_bias[b,h,j] =
 * sum_i P_ij (dP_ij - D_i) over the allowed pairs (the softcap factor does not
 * apply: the bias is added after the cap). The dynamic keep set is held fixed
 * (it changes only where two biases cross). Written for every key, 0 for keys
 * no query sees; also defined when key_bias is NULL (the gradient at zero).
 * Stream: stream-ordered on `stream` like every call. The bf16 path runs its
 * query-parallel (dQ) grid on a second stream that the library creates once
 * per calling host thread and device, forked from `stream` after the
 * preprocess (event record / wait) and joined back into `stream` before the
 * call returns, so work issued on `stream` afterwards sees every gradient and
 * CUDA graph capture on `stream` captures both grids. If that stream cannot be
 * created, both grids run on `stream`.
 */
int attn_bwd(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv,
             const void* q, const void* k, const void* v, const void* o,
             const void* dout, const float* lse, float scale,
             const gbattn_mask* mask, const gbattn_blocks* blocks, int deterministic,
             void* dq, void* dk, void* dv, float* dkey_bias,
             void* workspace, size_t workspace_bytes, gbattn_stream stream);

/* Workspace bytes attn_fwd_splitkv needs: num_splits partial outputs
 * [n,B,H,Sq,Dv] fp32 and partial LSEs [n,B,H,Sq] fp32 (0 when num_splits == 1). */
size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Sq, int Dv, int num_splits);

/*
 * attn_fwd_splitkv - decode-shaped forward ([FSA] split-KV forward, splits
 * 1/2/4/8/16 tested). The keys are cut into num_splits ranges of
 * L = ceil(Sk/num_splits) rounded up to 128 keys; each (b,h,split) streams
 * its K/V range once with 16-byte vector loads and writes a partial output and
 * LSE; a combine kernel merges them with the LSE-weighted rule of [PCB]
 * (num_splits == 1 writes O directly). bf16 only; mask kind NONE or CAUSAL,
 * no softcap or biases. 1 <= num_splits <= 64. With GQA (H / Hkv query
 * heads per key/value head) and at least 4 query rows per group, one CTA
 * streams each key/value row once for up to 8 (D = 128) or 16 (D = 64) query
 * rows of the group ([FA2C]'s pack_gqa).
 */
int attn_fwd_splitkv(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv,
                     const void* q, const void* k, const void* v, float scale,
                     const gbattn_mask* mask, int num_splits, void* o, float* lse,
                     void* workspace, size_t workspace_bytes, gbattn_stream stream);

/*
 * attn_fwd_splitkv_paged - attn_fwd_splitkv over a paged key/value cache
 * with a key count per sequence (the `page_table` / `seqused_k` arguments of
 * [FA2C]'s `_flash_attn_fwd`; the page layout is this library's choice).
 *   - k_cache, v_cache: [num_pages, Hkv, page_size, D] bf16: a page holds
 *     page_size consecutive keys of one sequence for every key/value head,
 *     each head's rows contiguous. page_size is a multiple of 64.
 *   - page_table: device [B, max_pages_per_seq] int32; key t of sequence b
 *     is row t % page_size of page page_table[b][t / page_size].
 *   - seqlens_k: device [B] int32, keys of sequence b (0 ..
 *     max_pages_per_seq * page_size). CAUSAL aligns query i with key
 *     i + seqlens_k[b] - Sq.
 *   - Splits cut each sequence's own keys (L = ceil(seqlens_k[b]/num_splits)
 *     rounded up to 128). With GQA and page_size a multiple of 128, the
 *     packed tensor-core path of attn_fwd_splitkv runs on the pages (one TMA
 *     tile load per 128 keys, the page looked up per tile).
 *   - A page index outside [0, num_pages) or a key count
 *     outside its range is not read: the kernel raises GBATTN_ERR_BLOCKS
 *     (gbattn_last_device_error) and the affected outputs are invalid.
 * Other arguments, workspace and status codes as attn_fwd_splitkv.
 */
int attn_fwd_splitkv_paged(int dtype, int B, int H, int Hkv, int Sq, int Dqk, int Dv,
                           const void* q, const void* k_cache, const void* v_cache,
                           int num_pages, int page_size, const int32_t* page_table,
                           int max_pages_per_seq, const int32_t* seqlens_k, float scale,
                           const gbattn_mask* mask, int num_splits, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, gbattn_stream stream);

/*
 * attn_fwd_splitkv_noalloc - attn_fwd_splitkv for callers that cannot
 * allocate device memory. The pages have no counterpart: this is a
 * convenience of this library, not a step of the method.
 *
 * Some callers only ever hold the buffers they are handed: a plug-in inside an
 * inference engine whose device memory all belongs to the engine's own
 * allocator, or a latency-critical decode loop that must not call cudaMalloc
 * once it runs (cudaMalloc can synchronise the device and stall other work).
 * They cannot provide the split workspace attn_fwd_splitkv asks for. This
 * entry point takes the same arguments minus the workspace and keeps the split
 * partials in a scratch array that the library holds in device memory: a
 * file-scope array of GBATTN_NOALLOC_SCRATCH_BYTES bytes, held on every GPU
 * that loads the library's decode code until the process exits. It calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *   - When the array's memory is committed: the CUDA runtime loads a device
 *     code module on a device when it is first used there (CUDA's default
 *     lazy module loading), and the array comes into being with its module.
 *     So the first call on each device (or the first split-KV call of any
 *     kind) can itself need 16 MiB of free device memory and fail with
 *     GBATTN_ERR_CUDA if there is none. Make one warm-up call on each device
 *     before your engine's allocator reserves the rest of the memory.
 *   - Limit: attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits) must
 *     not exceed GBATTN_NOALLOC_SCRATCH_BYTES; larger problems are rejected
 *     with GBATTN_ERR_WORKSPACE (use attn_fwd_splitkv with your own workspace).
 *     num_splits == 1 needs no scratch.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind. Calls
 *     whose GPU work overlaps (different streams, or several host threads)
 *     race on it and give wrong results: order them on one stream or
 *     synchronise between them.
 * Arguments, layouts, supported shapes and the other status codes are those of
 * attn_fwd_splitkv.
 */
#define GBATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
int attn_fwd_splitkv_noalloc(int dtype, int B, int H, int Hkv, int Sq, int Sk, int Dqk, int Dv,
                             const void* q, const void* k, const void* v, float scale,
                             const gbattn_mask* mask, int num_splits, void* o, float* lse,
                             gbattn_stream stream);

/*
 * gbattn_set_dkdv_cta_pair - which dK/dV kernel attn_bwd runs where the
 * CTA-pair kernel applies ("Enable 2CTA for SM100 block-sparse backward",
 * Summary: the 2-CTA backward over kv sub-tiles of a sparse block).
 *   The CTA-pair kernel runs a cluster of two CTAs per 256 keys whose
 *   tcgen05 MMAs span both SMs (M = 256 keys, each CTA holding half of the
 *   query-side operand). It applies to bf16 calls without gathered keys or an
 *   element table, with Dqk / Dv = 192 / 128 or 128 / 128, and with block
 *   lists whose sparse_n is a multiple of 256 (or no lists); other calls
 *   always run the one-CTA kernel. Both give the same gradients up to fp32
 *   summation order and both are deterministic.
 *   mode: 1 = the CTA-pair kernel where it applies, 0 = the one-CTA kernel,
 *   -1 = the library's default (the one measured faster on GB300).
 *   previous: if not NULL, receives the mode in effect before the call.
 *   Process-wide; takes effect for calls issued after it returns.
 * Returns GBATTN_OK, or GBATTN_ERR_ARG for a mode outside -1..1 (nothing
 * changes).
 */
int gbattn_set_dkdv_cta_pair(int mode, int* previous);

/* Synchronises `stream`, then returns and clears the device-side error word
 * of the current device: GBATTN_OK, GBATTN_ERR_TIMEOUT (a bounded wait inside
 * a kernel ran out; the kernel returned early and its outputs are invalid) or
 * GBATTN_ERR_BLOCKS (a kernel met an out-of-range list entry and skipped it). */
int gbattn_last_device_error(gbattn_stream stream);

/* Static, human-readable text for a status code. */
const char* gbattn_strerror(int status);

/* ABI version: 100 * major + minor. */
int gbattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GBATTN_H */
