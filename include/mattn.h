/*
 * mattn.h - C ABI of the masked-attention library (libmattn.so) for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The library computes fused scaled-dot-product attention with an element-wise
 * score modification and a mask, in one pass over key/value tiles with an
 * online softmax, so the Sq x Skv score matrix never reaches device memory:
 *
 *   s[b,h,i,j] = scale * <q[b,h,i,:], k[b,hk,j,:]>            hk = h / (Hq/Hkv)
 *   s'         = score_mod(s, b, h, i, j)                       (before softmax)
 *   O[b,h,i,:] = sum over kept j of softmax_j(s') * v[b,hk,j,:]
 *   LSE[b,h,i] = ln sum over kept j of exp(s'[b,h,i,j])
 *
 * Sources: the FlexAttention page (section "FlexAttention": a user function
 * score_mod(score, b, h, q_idx, kv_idx) modifies every score before the
 * softmax; the variant list: causal, relative position, ALiBi, sliding window,
 * PrefixLM, document masking; the item on exploiting mask sparsity; section
 * "Performance": a deterministic backward that recomputes intermediates) and
 * the Online-Softmax/FlashAttention page (abstract: 3-pass safe softmax,
 * 2-pass online softmax, 1-pass FlashAttention).
 *
 * Conventions for every entry point:
 *  - Buffers are caller-owned. Tensor arguments are DEVICE pointers; structs
 *    (attn_params, attn_block_mask) live in HOST memory. The library allocates
 *    no device memory on any call.
 *  - Layout: contiguous [B, H, S, D], D innermost. Base pointers of q, k, v,
 *    o, dO, dq, dk, dv must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). Argument errors are returned before anything is launched. A
 *    failed launch returns ATTN_ERR_CUDA. Device-side failures (a bounded wait
 *    that ran out) are written to the status word and read back with
 *    attn_check_status().
 *  - No C++ exception crosses this boundary. The functions are thread-safe.
 */
#ifndef MATTN_H_
#define MATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*` */

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,        /* NULL pointer, bad size, inconsistent shapes */
  ATTN_ERR_UNSUPPORTED = 2,        /* valid but not built: D, dtype, tails, variant */
  ATTN_ERR_MISALIGNED = 3,         /* a tensor base pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE_TOO_SMALL = 4,/* the caller's buffer is smaller than required */
  ATTN_ERR_CUDA = 5,               /* a CUDA runtime call or a launch failed */
  ATTN_ERR_TIMEOUT = 6             /* a device-side bounded wait ran out */
} attn_status;

/* Variant: OR of the bits below; 0 = full (bidirectional) attention with the
 * identity score_mod. Mask terms combine as
 *   keep(b,i,j) = (CAUSAL: j <= i) AND (WINDOW: i - j < window)
 *                 AND (DOCUMENT: doc_id[b][i] == doc_id[b][j])
 *                 OR  (PREFIX: j < prefix_len[b])
 * with absent AND-terms true and an absent PREFIX false. i and j are absolute
 * positions: i = q_offset + query row, j = kv_offset + key column (both
 * offsets 0 unless the call is one shard of a longer sequence, see
 * attn_params and attn_combine).
 * Score terms apply in this order: s <- scale * q.k; ALIBI: s <- s - slope_h
 * * (i - j); RELBIAS: s <- s + rel_bias[h][i - j + Skv - 1]; SOFTCAP:
 * s <- softcap * tanh(s / softcap). */
enum {
  ATTN_MASK_CAUSAL = 1u << 0,   /* FlexAttention page, "Causal Mask" */
  ATTN_MASK_WINDOW = 1u << 1,   /* "Sliding Window + Causal" (1024 tokens there) */
  ATTN_MASK_DOCUMENT = 1u << 2, /* variant list: document masking */
  ATTN_MASK_PREFIX = 1u << 3,   /* variant list: PrefixLM (prefix is bidirectional) */
  ATTN_SCORE_ALIBI = 1u << 8,   /* variant list: ALiBi; slope_h = 2^(-8(h+1)/Hq) */
  ATTN_SCORE_SOFTCAP = 1u << 9, /* "Soft-capping" section (Gemma 2, Grok-1) */
  ATTN_SCORE_RELBIAS = 1u << 10 /* relative position encoding: the score is adjusted by
                                   the query-key distance, from a per-head table the
                                   call captures (no S x S tensor); forward only */
};
#define ATTN_MASK_BITS 0x0Fu
#define ATTN_SCORE_BITS 0x700u

enum { ATTN_BF16 = 0, ATTN_F32 = 1 };

/* Tile size of the block mask and of the kernels (query rows x key columns). */
#define ATTN_TILE 128

/* Block mask: per (batch, 128-row query tile) the ascending lists of
 * 128-column key tiles that are FULL (every pair kept: no mask evaluated) or
 * PARTIAL (some pairs kept: the mask is evaluated per element); EMPTY tiles
 * are skipped (FlexAttention page: exploiting the sparsity of the mask). The
 * mask does not depend on the head, so one list serves every head. All
 * pointers below point into the caller's device buffer given to
 * build_block_mask(); this host struct only describes it.
 *   full_cnt, part_cnt  int32 [B][nq]
 *   full_idx, part_idx  int32 [B][nq][nkv]  (first *_cnt entries valid)
 *   order               int32 [B*nq]: b*nq+qt by descending full+part count
 *                       (ties by ascending index): longest work first
 * The t_* members hold the transposed lists (per key tile, its query tiles,
 * [B][nkv] and [B][nkv][nq]) when built with transposed = 1, else NULL;
 * t_order lists their rows batch element by batch element (ascending b),
 * within one by descending full+part count (ties by ascending index). */
typedef struct attn_block_mask {
  int B, Sq, Skv;
  int nq, nkv;
  unsigned variant;      /* mask bits it was built for */
  int window;            /* parameters it was built for */
  const int* doc_id;
  const int* prefix_len;
  const int* full_cnt;
  const int* part_cnt;
  const int* full_idx;
  const int* part_idx;
  const int* order;
  const int* t_full_cnt;
  const int* t_part_cnt;
  const int* t_full_idx;
  const int* t_part_idx;
  const int* t_order;
  int q_offset, kv_offset;  /* position offsets it was built for */
  int doc_len;              /* row length of doc_id it was built for */
} attn_block_mask;

/* Parameters of a call (host struct). */
typedef struct attn_params {
  int dtype;                   /* ATTN_BF16 or ATTN_F32: type of q, k, v, o, do, dq, dk, dv */
  float scale;                 /* multiplies q.k, > 0; 0 selects 1/sqrt(D) */
  int window;                  /* ATTN_MASK_WINDOW: keys with i - j < window; >= 1 */
  float softcap;               /* ATTN_SCORE_SOFTCAP: cap c > 0 */
  const float* alibi_slopes;   /* ATTN_SCORE_ALIBI: device fp32 [Hq], or NULL for 2^(-8(h+1)/Hq) */
  const int* doc_id;           /* ATTN_MASK_DOCUMENT: device int32 [B][doc_len], indexed
                                  by absolute position */
  const int* prefix_len;       /* ATTN_MASK_PREFIX: device int32 [B] */
  const attn_block_mask* block_mask; /* from build_block_mask() for the same mask, or NULL:
                                        then every key tile allowed by the causal bound is
                                        visited with the mask evaluated per element */
  int* status;                 /* device int32 status word, or NULL for the library's own */
  unsigned long long timeout_ns; /* limit of each device-side wait; 0 = 4 s */
  const float* rel_bias;       /* ATTN_SCORE_RELBIAS: device fp32 [Hq][Sq + Skv - 1]; entry
                                  d + Skv - 1 is added to the score of a query-key pair at
                                  distance d = i - j (4-byte aligned). Not differentiated:
                                  attn_bwd returns ATTN_ERR_UNSUPPORTED with this bit */
  unsigned fault_inject;       /* 0 in normal use. ATTN_FAULT_NO_LOADS: the tensor-core
                                  kernels' load warp issues no copy, so every wait for data
                                  runs out after timeout_ns and the call reports
                                  ATTN_ERR_TIMEOUT (tests the bounded-wait path; no GPU
                                  fault is involved) */
  /* Paged K/V cache (variant list: PagedAttention), bf16 forward only. NULL
   * page_table: k and v are contiguous [B,Hkv,Skv,D]. Otherwise k and v are
   * page pools [num_pages][Hkv][page_size][D] and key j of batch b is row
   * j % page_size of page page_table[b * pages_per_seq + j / page_size].
   * page_size is 16, 32, 64 or 128; pages_per_seq * page_size >= Skv. Rows
   * of the last page past Skv are read (and masked): they must hold finite
   * values. A page index outside [0, num_pages) reads zeros. Not combined
   * with ATTN_SCORE_RELBIAS (ATTN_ERR_UNSUPPORTED). */
  const int* page_table;       /* device int32 [B][pages_per_seq], or NULL */
  int page_size;
  int pages_per_seq;
  int num_pages;
  /* Shards of a longer sequence (FlexAttention page, variant list: sliding
   * window + document masking + causal + context parallel): query row r and
   * key column c of this call sit at absolute positions q_offset + r and
   * kv_offset + c, which every mask term, the ALiBi bias and the document ids
   * use. Results over disjoint key shards merge with attn_combine(). >= 0.
   * Forward, backward and block mask; not combined with ATTN_SCORE_RELBIAS. */
  int q_offset;
  int kv_offset;
  /* Row length of doc_id: 0 selects L = max(q_offset + Sq, kv_offset + Skv);
   * otherwise >= L (e.g. the whole sequence's length when the call is one
   * shard of it). */
  int doc_len;
} attn_params;

#define ATTN_FAULT_NO_LOADS 1u

/* Forward: O = softmax(score_mod(scale*QK^T) under the mask) V and LSE.
 *   q [B,Hq,Sq,D], k and v [B,Hkv,Skv,D], o [B,Hq,Sq,D] (dtype p->dtype),
 *   lse fp32 [B,Hq,Sq] (natural log; -inf for a row with no kept key, whose
 *   O row is 0).
 * Supported: D in {64, 128}; Hq % Hkv == 0 (GQA: query head h reads key/value
 * head h / (Hq/Hkv)); any Sq, Skv >= 1 for both ATTN_BF16 (tcgen05
 * tensor-core kernel: a last tile that runs past Sq or Skv reads zero-filled
 * rows, its extra keys are masked and its extra query rows are not stored)
 * and ATTN_F32 (fp32 FFMA kernel). Returns ATTN_ERR_UNSUPPORTED for anything
 * else. */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Sq, int Skv, int D,
                     unsigned variant, const attn_params* p, struct CUstream_st* stream);

/* Decode: a few new query rows per sequence against a long key/value cache
 * (FlexAttention page, variant list: PagedAttention, alone and with a
 * sliding window). Same arguments, layouts and results as attn_fwd for
 * ATTN_BF16, D = 64 or 128, with (Hq / Hkv) * Sq <= 16: the query rows of all
 * query heads that share a key/value head are computed together, so each
 * key and value row is read from memory once. K and V are contiguous or a
 * paged cache (attn_params page_table etc., page_size 16, 32, 64 or 128); a
 * page index outside [0, num_pages) reads as zeros. Every mask and score term
 * is supported; for a new token at absolute position P, pass q_offset = P
 * so the causal and window terms see it. p->block_mask is not used.
 * The keys are split across CTAs when that gives more parallelism: the
 * splits' partial results (fp32) go to `workspace` (device, 256-byte aligned,
 * attn_decode_workspace_bytes() bytes for the full split count) and are
 * merged into o and lse by the online-softmax merge. A smaller workspace (or
 * NULL) means fewer splits (none with NULL). Asynchronous on `stream`;
 * argument errors before any launch; ATTN_ERR_UNSUPPORTED for other dtypes,
 * D or row counts, or B * Hkv > 65535. */
attn_status attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D,
                        unsigned variant, const attn_params* p,
                        void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/* Bytes of workspace attn_decode() uses for its full split count on the
 * current device (0 when it does not split the keys). */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D);

/* Merge of partial results over disjoint key sets, e.g. the key/value shards
 * of context-parallel attention (FlexAttention page, variant list: ... +
 * context parallel). It is the merge step of the online softmax
 * (Online-Softmax/FlashAttention page, 2-pass online softmax: partial maxima
 * and sums combine as m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m)) applied
 * to whole results, each normalised by its own sum:
 *   LSE = ln sum_k exp(LSE_k),   O = sum_k exp(LSE_k - LSE) O_k
 * and a row with no kept key in any part (every LSE_k = -inf) gets O = 0 and
 * LSE = -inf. A part whose LSE_k is -inf is not read.
 *   o_parts   device [n_parts][rows][D] of `dtype` (ATTN_BF16 or ATTN_F32),
 *             part k = the forward output of the same queries against key
 *             set k (rows = B * H * S in [B, H, S, D] order)
 *   lse_parts device fp32 [n_parts][rows]
 *   o, lse    device [rows][D] of `dtype` and fp32 [rows]; they must not
 *             overlap the parts.
 * D is 64 or 128; n_parts >= 1; 16-byte aligned tensors. Asynchronous on
 * `stream`. ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED / ATTN_ERR_MISALIGNED
 * before any launch. */
attn_status attn_combine(const void* o_parts, const float* lse_parts, int n_parts,
                         long long rows, int D, int dtype, void* o, float* lse,
                         struct CUstream_st* stream);

/* Jagged batches (FlexAttention page, variant list: irregular tensors): n
 * sequences packed back to back with no padding, cu_seqlens (device int32
 * [n + 1]: 0 = cu[0] <= cu[1] <= ... <= cu[n] = total) their cumulative
 * lengths. Writes doc_id (device int32 [total]) = the index of the sequence
 * each packed position belongs to. With B = 1, S = total and
 * ATTN_MASK_DOCUMENT (plus ATTN_MASK_CAUSAL etc.) the forward, backward and
 * block mask then attend within each sequence only. Asynchronous on
 * `stream`; ATTN_ERR_INVALID_ARG for n < 1, total < 0 or null pointers. The
 * lengths are not validated on the device: non-monotone input gives
 * undefined ids. */
attn_status attn_doc_ids_from_seqlens(const int* cu_seqlens, int n, int total, int* doc_id,
                                      struct CUstream_st* stream);

/* Bytes of device buffer build_block_mask() needs (256-byte aligned pieces). */
size_t attn_block_mask_bytes(int B, int Sq, int Skv, int transposed);

/* Classifies every (query tile, key tile) pair as full, partial or empty
 * under the mask bits of `variant` (score bits are ignored) and writes the
 * lists into `buf` (device, `bytes` long, 256-byte aligned). Fills `*out`
 * (host) with pointers into `buf`. The result is exact: a tile is full iff
 * every pair in it is kept and empty iff none is. */
attn_status build_block_mask(unsigned variant, const attn_params* p, int B, int Sq, int Skv,
                             void* buf, size_t bytes, int transposed, attn_block_mask* out,
                             struct CUstream_st* stream);

/* Bytes of fp32 workspace attn_bwd() needs: B*Hq*Sq*4 (the row terms
 * Delta_i = <dO_i, O_i>). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq);

/* Bytes of workspace for attn_bwd()'s fp16 path: the row terms, then fp16
 * copies of q, k, v and dO (about 2 (B Hq Sq + B Hkv Skv) D * 2 bytes more).
 * A call given at least this much, with Sq and Skv multiples of 128, no
 * position offsets and no relative-position bias, converts its inputs to fp16
 * (recording their largest |x|) and, where every |x| <= 60000 and
 * 2 D max|dO| max|V| <= 60000, computes the gradients from fp16 operands: each
 * product of a probability or dS term with an input is then one tensor-core
 * product instead of the bf16 path's two (the bf16 value and its rounding
 * remainder). Otherwise, and with a smaller workspace, the bf16 path runs.
 * Both meet the same bound. */
size_t attn_bwd_workspace_bytes_f16(int B, int Hq, int Hkv, int Sq, int Skv, int D);

/* Backward of the forward above (FlexAttention page, "Performance": a
 * deterministic backward that recomputes intermediates instead of storing
 * them): from q, k, v, o, lse and dO computes
 *   dq [B,Hq,Sq,D], dk and dv [B,Hkv,Skv,D] (dtype p->dtype; with GQA, dk and
 *   dv sum over the query heads of their group).
 * `workspace` is device memory of attn_bwd_workspace_bytes() bytes, or of
 * attn_bwd_workspace_bytes_f16() bytes for the fp16 path (see there). No
 * atomics: results are bitwise reproducible. Supported: ATTN_BF16, D = 128 and
 * 64, any Sq, Skv >= 1 (a last tile that runs past Sq or Skv reads zero rows,
 * its padding keys are masked and its padding rows are not stored); a block
 * mask built with transposed = 1 (or NULL); position offsets (attn_params
 * q_offset, kv_offset), with a block mask built for the same offsets: the
 * gradients of this call's own attention (its o and lse over its keys); the
 * relative-position bias (a constant of the call: no gradient flows to the
 * table), not together with offsets. Not supported (ATTN_ERR_UNSUPPORTED):
 * paged K/V. */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes,
                     int B, int Hq, int Hkv, int Sq, int Skv, int D,
                     unsigned variant, const attn_params* p, struct CUstream_st* stream);

/* attn_bwd for callers that cannot allocate device memory. The page this
 * library follows has no counterpart: it exists for code that is handed its
 * tensors but has no way to obtain a workspace (a framework that owns every
 * device allocation and forbids raw cudaMalloc, a plug-in without an
 * allocator). Same arguments and results as attn_bwd without `workspace`:
 * the Delta row terms live in a fixed array inside the library (8 MiB per
 * GPU that loads it, held until the process exits), so B*Hq*Sq may be at most
 * 2,097,152; larger problems return ATTN_ERR_WORKSPACE_TOO_SMALL before
 * anything runs (every other argument is checked first, with no CUDA call).
 * No cudaMalloc, cudaFree or other allocating call is made. The first call
 * on a device looks up the array's device address and keeps it (make that
 * call before any stream capture); the address belongs to the device's
 * primary context, so after cudaDeviceReset the entry point must not be
 * called again in the same process. Every call shares the array, which keeps the
 * last call's contents (none needs to start at zero); calls that overlap on
 * the GPU race on it. */
attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dO, void* dq, void* dk, void* dv,
                             int B, int Hq, int Hkv, int Sq, int Skv, int D,
                             unsigned variant, const attn_params* p, struct CUstream_st* stream);

/* Synchronises `stream`, reads the device status word (`status_dev`, or the
 * library's own when NULL), resets it to 0 and returns it as an attn_status. */
attn_status attn_check_status(int* status_dev, struct CUstream_st* stream);

/* Static string naming a status code. */
const char* attn_status_str(attn_status s);

/* Name of the CUDA runtime error behind the calling thread's most recent
 * ATTN_ERR_CUDA (e.g. "cudaErrorLaunchOutOfResources"), or "cudaSuccess"
 * if none occurred on this thread. Static string; makes no CUDA call that
 * can fail. */
const char* attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MATTN_H_ */
