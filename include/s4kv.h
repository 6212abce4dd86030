/*
 * s4kv.h — C ABI of the GB300 (sm_103a) int4 KIVI-style paged KV cache and the
 * decode-attention kernel that reads it.
 *
 * What the library computes (sources: the web pages describing the method).
 *  - "4.4 KV Cache 量化", section 3.1: keys are quantized per channel — one
 *    (scale, min) per channel over each group of G consecutive tokens; values
 *    are quantized per token — one (scale, min) per token over each group of Gv
 *    channels. Inside a group the mapping is asymmetric, from its minimum and
 *    maximum; 4-bit codes give 16 levels.
 *  - same page, section 3.2: new key tokens wait in a full-precision residual
 *    until a key group is full, and the full group is then quantized as a batch
 *    into the history; the value residual is a sliding window of the newest R
 *    tokens, each arrival pushing the oldest one out into the quantized history.
 *    Residual and history both take part in attention.
 *  - same page, section 1: fixed-size physical pages (PagedAttention) and
 *    quantization stack: pages remove waste, quantization shrinks each element.
 *  - same page, section 2: attention P = softmax(Q K^T / sqrt(d)), output P V.
 *  - "给 KV cache 减肥", section 3.1: compress before the write to HBM, restore
 *    when the next query reads.
 *  - "S4 KV" product page: head_dim 128, standard attention; anything else fails
 *    at start-up rather than producing wrong output.
 *
 * Quantizer (exact; the GPU matches it bit for bit):
 *     mn = min(x) + 0.0f, mx = max(x) + 0.0f          (fp32; -0 becomes +0)
 *     s  = (mx - mn) / 15.0f                          (IEEE sub, then IEEE div)
 *     c  = s == 0 ? 0 : clamp(round_half_even((x - mn) / s), 0, 15)
 *     restored x^ = fmaf(c, s, mn)
 *
 * Conventions.
 *  - Every function returns an int status (S4KV_OK = 0, else an S4KV_ERR_*).
 *  - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned. The library owns only a small host handle.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Device calls are asynchronous on it and never synchronise, except
 *    s4kv_cache_create (zero-fills the header) and s4kv_get_status.
 *  - Device-side faults of the caller's data (a block-table entry out of range,
 *    a sequence length that disagrees with the cache, a slot out of range) never
 *    trap: the kernel skips the affected work item and records the error in a
 *    status word inside the pool; s4kv_get_status reports and clears it.
 *  - Only one configuration is supported: head_dim 128, page_size 16, G 32,
 *    Gv 32, fp16 or bf16 inputs, GQA group (H_q / H_kv) 1..8. Anything else
 *    fails with S4KV_ERR_UNSUPPORTED at create (or at the call for H_q).
 *
 * Physical format of one (layer, page, kv head) record with 4-bit codes (the
 * default): 3072 bytes, 16 tokens.
 *   [0, 1024)    key codes       [1024, 1536) key scale/min (fp32)
 *   [1536, 2560) value codes     [2560, 3072) value scale/min (fp32)
 *   Lane L = 4a + b with a in 0..7, b in 0..3; tau = token within the page.
 *   Key codes: 32-bit word (kk, L), kk in 0..7, at byte (kk/4)*512 + L*16 +
 *     (kk%4)*4 holds channels c_j = 32b + 4kk + j of tokens a (low nibbles) and
 *     a + 8 (high nibbles); its byte 0 holds c_0, byte 1 c_2, byte 2 c_1,
 *     byte 3 c_3. (This is the A-operand fragment order of an m16n8k16 MMA with
 *     tokens as rows: one 32-bit word per lane per 16-channel slice.)
 *   Key scale/min: a key group's 32 tokens fill logical pages 2m and 2m+1; page
 *     2m+j holds channels 64j..64j+63. Channel 64j + 32u + 4i + e (u 0..1,
 *     i 0..7, e 0..3): scale at byte 1024 + (2i+u)*16 + 4e, min 256 bytes later.
 *   Value codes: word (mt, L), mt in 0..7, at byte 1536 + (mt/4)*512 + L*16 +
 *     (mt%4)*4; low nibble = channel 16mt + a, high nibble = channel 16mt + a + 8;
 *     byte 0 holds token 2b, byte 1 token 2b+8, byte 2 token 2b+1, byte 3 token
 *     2b+9. (A-operand order with channels as rows, tokens as columns; each
 *     token owns whole bytes, so single tokens are written without
 *     read-modify-write.)
 *   Value scale/min: token tau = 2b + r + 8w (r, w in 0..1) is entry e = r + 2w
 *     of column b; the scale of its channel group k (channels 32k..32k+31) is at
 *     byte 2560 + ((2k)*4 + b)*16 + 4e, the min at 2560 + ((2k+1)*4 + b)*16 + 4e.
 *   Bytes of tokens not yet quantized are undefined.
 * 2-bit records (cfg.bits = 2), 2048 bytes: [0, 512) key codes, [512, 1024)
 *   key scale/min, [1024, 1536) value codes, [1536, 2048) value scale/min; the
 *   scale/min regions are laid out as above. A byte holds four 2-bit codes;
 *   "position p" is bits 2p .. 2p+1.
 *   Key codes: word (kp, L), kp in 0..3, at byte L*16 + kp*4 covers the channels
 *     of slices kk = 2kp and 2kp+1; byte 0 <- c_0, byte 1 <- c_2, byte 2 <- c_1,
 *     byte 3 <- c_3; position 0 <- (token a, 2kp), 1 <- (token a+8, 2kp),
 *     2 <- (token a, 2kp+1), 3 <- (token a+8, 2kp+1).
 *   Value codes: word (mp, L), mp in 0..3, at byte 1024 + L*16 + mp*4; bytes
 *     hold tokens as above (0 <- 2b, 1 <- 2b+8, 2 <- 2b+1, 3 <- 2b+9); position
 *     q <- channel 32*mp + 8*q + a.
 * FP8 E4M3 records (cfg.bits = 8; "4.4 KV Cache 量化", sections 4.1 and 4.2:
 *   the fp8_e4m3 KV type, one scale per attention head, 1.0 unless calibrated),
 *   4096 bytes: [0, 2048) keys, [2048, 4096) values, one byte per element, no
 *   metadata and no rings: each token is written to its page on arrival as
 *   e4m3(x / scale) (x / scale rounded to fp32, then nearest-even to E4M3,
 *   saturating at +-448) and restored as value(code) * scale. Word (kp, L),
 *   kp in 0..3, is the 16 bytes at kp*512 + L*16 of a half.
 *   Keys: bytes 8u .. 8u+7 of word (kp, L) hold slice kk = 2kp + u (channels
 *     c_j = 32b + 4kk + j): byte 8u + 4*(j/2) + 2*hi + (j%2) is token a + 8*hi
 *     of channel c_j.
 *   Values: bytes 8u .. 8u+7 of word (kp, L) hold channels 16mt + a + 8*up of
 *     tile mt = 2kp + u: byte 8u + 4w + 2*up + r is token 2b + r + 8w.
 *   (Each byte pair is one f16x2 MMA operand register after conversion.)
 *   Bytes of a page past the sequence's length are undefined.
 * Residual rings (cache dtype): key ring [slot][kv head][32][128], token t at
 *   row t mod 32; value ring [slot][kv head][R][128], token t at row t mod R.
 * Canonical state of a sequence of length T: keys of tokens < 32*floor(T/32)
 *   and values of tokens < max(0, T - R) are quantized in pages; the rest sit in
 *   the rings. It depends only on the tokens and T, never on how the appends
 *   were chunked.
 */
#ifndef S4KV_H
#define S4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  S4KV_OK = 0,
  S4KV_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size or index; also
                                    any call that launches work (append, attention,
                                    decode step, dequant) while the current device is
                                    not the one the cache was created on */
  S4KV_ERR_UNSUPPORTED = 2,      /* a shape this build does not implement */
  S4KV_ERR_CUDA = 3,             /* a CUDA runtime call failed */
  S4KV_ERR_POOL_TOO_SMALL = 4,   /* pool_bytes < s4kv_cache_bytes() */
  S4KV_ERR_DEVICE = 5,           /* a kernel found bad caller data (status word) */
  S4KV_ERR_DEVICE_TIMEOUT = 6,   /* a bounded device wait ran out */
  S4KV_ERR_WORKSPACE_TOO_SMALL = 7
};

enum { S4KV_F16 = 0, S4KV_BF16 = 1, S4KV_F32 = 2 };

/* Device status detail codes (second word of the status area). */
enum {
  S4KV_DEV_BAD_PAGE = 1,       /* block-table entry outside [0, num_pages) */
  S4KV_DEV_BAD_LENGTH = 2,     /* length disagrees with the slot's stored length */
  S4KV_DEV_BAD_SLOT = 3,       /* slot id outside [0, max_slots) */
  S4KV_DEV_BAD_TABLE = 4,      /* table too narrow for the sequence */
  S4KV_DEV_BAD_CU = 5,         /* cu_new not non-decreasing / total mismatch */
  S4KV_DEV_TIMEOUT = 6         /* an mbarrier wait exceeded its limit */
};

typedef struct {
  int num_layers;    /* layers sharing the pool (one page region per layer) */
  int num_pages;     /* physical pages per layer */
  int page_size;     /* P, tokens per page: must be 16 */
  int num_kv_heads;  /* H_kv, 1..64 */
  int head_dim;      /* d: must be 128 (fail-fast otherwise) */
  int group_k;       /* G, tokens per key group: must be 32 */
  int group_v;       /* Gv, channels per value group: must be 32 */
  int residual_v;    /* R, value sliding window: 1..1024 */
  int max_slots;     /* sequence slots (residual rings), 1..65536 */
  int dtype;         /* S4KV_F16 or S4KV_BF16: the K/V/Q input format */
  int bits;          /* code width: 4 (0 means 4) or 2, the pages' own KIVI
                        settings; 8 selects FP8 E4M3 pages instead (below) */
} s4kv_config;

typedef struct s4kv_cache s4kv_cache;

/* Byte offsets of everything inside the pool (for byte-level checks). */
typedef struct {
  size_t pool_bytes;
  size_t status_offset;      /* int32 status, int32 detail, int32 arg */
  size_t lens_offset;        /* int32 [num_layers][max_slots]: stored lengths */
  size_t layer_offset;       /* first layer region */
  size_t layer_stride;
  size_t page_stride;        /* bytes per physical page (all kv heads) */
  size_t record_bytes;       /* bytes per (page, kv head): 3072 */
  size_t kcode_offset, kmeta_offset, vcode_offset, vmeta_offset;  /* in a record */
  size_t kring_offset;       /* inside a layer region */
  size_t kring_slot_stride, kring_head_stride, kring_row_stride;
  size_t vring_offset;
  size_t vring_slot_stride, vring_head_stride, vring_row_stride;
  size_t scale_offset;       /* FP8 pools: float [num_layers][2][H_kv], key scales
                                then value scales; 0 for KIVI pools */
} s4kv_layout;

/* Memory ledger for B sequences of T tokens over all layers (section 1 of the
 * KV-cache quantization page: M_KV = 2 L B T H_KV d b). */
typedef struct {
  double fp16_equiv_bytes;   /* M_KV at b = 2 bytes */
  double code_bytes;         /* 4-bit codes only: M_KV(b = 0.5) */
  double meta_bytes;         /* fp32 scale + min of key and value groups */
  double residual_bytes;     /* the rings of B slots */
  double paged_bytes;        /* ceil(T / P) pages * record bytes * H_kv * L * B */
} s4kv_kv_bytes_report;

/* Pool size for `cfg`, and the paged bytes per (token, kv head) (192).
 * Errors: INVALID_ARG for null pointers or nonsensical sizes, UNSUPPORTED for a
 * shape this build does not implement (head_dim != 128 first of all). */
int s4kv_cache_bytes(const s4kv_config* cfg, size_t* pool_bytes, size_t* bytes_per_token_head);

/* Capacity: how many tokens of KV fit in `budget_bytes` of device memory for
 * this configuration ("how many KV tokens fit", the question the pages' memory
 * formula M_KV = 2 L B T H_KV d b answers for a cache). The largest page count
 * whose pool (cfg with that num_pages; the rings of cfg.max_slots slots, the
 * lengths and the status area included) is <= budget_bytes; *tokens = 16 *
 * pages (token positions, each over every layer and kv head), *pages = pages.
 * cfg.num_pages is ignored. Errors: those of s4kv_cache_bytes; INVALID_ARG for
 * null outputs or a negative budget. 0 tokens when not even one page fits. */
int s4kv_capacity_tokens(const s4kv_config* cfg, double budget_bytes, long long* tokens, long long* pages);

/* Binds a cache to caller-allocated device memory `d_pool` (>= s4kv_cache_bytes,
 * 256-byte aligned) and zero-fills the status area and stored lengths
 * (synchronous). The pool stays owned by the caller and must outlive the cache.
 * Page and ring contents are not touched: a slot starts empty when it is first
 * appended to with seq_lens_before = 0. */
int s4kv_cache_create(const s4kv_config* cfg, void* d_pool, size_t pool_bytes, s4kv_cache** out);

/* FP8 pools (cfg.bits = 8): sets the key and value scales of one layer, host
 * arrays k_scale[H_kv], v_scale[H_kv], each finite and > 0 (INVALID_ARG
 * otherwise; UNSUPPORTED on a KIVI pool). Scales start at 1.0 at create. The
 * call synchronises `stream` (work queued before it keeps the old scales),
 * then copies the 2 H_kv floats synchronously. Tokens appended earlier keep
 * the codes they were written with: set a layer's scales before its first
 * append. */
int s4kv_set_fp8_scales(s4kv_cache* cache, int layer, const float* k_scale, const float* v_scale, void* stream);

/* Frees the host handle only. */
int s4kv_cache_destroy(s4kv_cache* cache);

int s4kv_get_layout(const s4kv_cache* cache, s4kv_layout* out);

/* Write side (section 3.2): appends new tokens of n sequences to one layer.
 *   k, v             [num_new_tokens][H_kv][128] cache dtype, ragged by sequence:
 *                    sequence i owns rows [cu_new[i], cu_new[i+1]).
 *   cu_new           int32 [n+1], non-decreasing, cu_new[0] = 0,
 *                    cu_new[n] = num_new_tokens.
 *   slot_ids         int32 [n] residual slot of each sequence (NULL: slot = i);
 *                    slots must be distinct within one call.
 *   seq_lens_before  int32 [n] current length T0 of each sequence; 0 starts the
 *                    slot afresh, any other value must equal the slot's stored
 *                    length (else S4KV_DEV_BAD_LENGTH).
 *   block_table      int32 [n][bt_stride]: row i maps logical page j of sequence
 *                    i to a physical page; it must already cover
 *                    ceil((T0 + new) / 16) pages.
 * Effect: every key group completed by the new tokens is quantized into its two
 * pages, every value token leaving the R-window is quantized into its page
 * slot, the remaining new tokens go to the rings. Afterwards the slot is in the
 * canonical state of length T0 + new. One kernel launch. */
int s4kv_append(s4kv_cache* cache, int layer, const void* k, const void* v, int num_new_tokens,
                const int32_t* cu_new, const int32_t* slot_ids, const int32_t* seq_lens_before,
                const int32_t* block_table, int bt_stride, int n, void* stream);

/* Scratch needed by s4kv_decode_attention for B sequences (two partial results
 * per worker warp; it depends on B, the GQA group and the device, not on the
 * lengths; max_seq_len is accepted for symmetry with the decode call). */
int s4kv_decode_workspace_bytes(const s4kv_cache* cache, int B, int num_q_heads, int max_seq_len,
                                size_t* bytes);

/* Read side (section 2): one decode query per sequence over the quantized
 * history plus the residual.
 *   B           sequences of the call, 0..4096.
 *   q           [B][num_q_heads][128] cache dtype; query head j reads KV head
 *               j / (num_q_heads / H_kv).
 *   block_table int32 [B][bt_stride] (row b for sequence b).
 *   seq_lens    int32 [B]: T_b, which must equal the slot's stored length
 *               (attention covers every appended token, the newest included);
 *               0 gives a zero output row.
 *   slot_ids    int32 [B] or NULL (slot = b).
 *   sm_scale    softmax scale; <= 0 means 1/sqrt(128).
 *   out         [B][num_q_heads][128] in out_dtype (S4KV_F32 or the cache dtype).
 *   workspace   device scratch of >= s4kv_decode_workspace_bytes(B, H_q,
 *               max_seq_len) bytes, where max_seq_len bounds every seq_lens[b];
 *               any contents; used only during the call (stream-ordered).
 * Two kernel launches on `stream`: split-K over the sequence with online
 * softmax (each split that does not cover a whole (sequence, kv head) leaves a
 * partial in the workspace), then a small kernel that combines those partials;
 * it is launched as a programmatic dependent of the first, so it is scheduled
 * while the first drains and starts reading once it has completed. */
int s4kv_decode_attention(s4kv_cache* cache, int layer, const void* q, int num_q_heads,
                          const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                          const int32_t* slot_ids, int B, float sm_scale, void* out,
                          int out_dtype, void* workspace, size_t ws_bytes, int max_seq_len,
                          void* stream);

/* Causal attention of a chunk of query tokens per sequence: the tokens of a
 * chunked-prefill step, or the draft tokens a speculative step verifies.
 * The pages write attention as P = softmax(QK^T / sqrt d), output P V
 * ("给 KV cache 减肥" section 2), with the residual rows and the quantized
 * history taking part together (section 3.2); a chunk of queries is read here
 * as the causal form of that over the state after the chunk was appended.
 *   q            [B][num_q_tokens][num_q_heads][128], cache dtype, 16-byte
 *                aligned: the queries of the last num_q_tokens positions.
 *   num_q_tokens nq, 1..16 (and <= R on KIVI pages); nq * (num_q_heads / H_kv)
 *                <= 96. KIVI and FP8 pools alike.
 *   seq_lens[b]  T_b >= nq, equal to the slot's appended length (the chunk's
 *                own tokens included).
 *   out          [B][num_q_tokens][num_q_heads][128] in out_dtype.
 * Query i of sequence b sits at position T_b - nq + i and attends to tokens
 * 0 .. T_b - nq + i (a causal mask over the chunk). Other arguments, the
 * workspace rule and the errors are those of s4kv_decode_attention; T_b < nq
 * is reported as S4KV_DEV_BAD_LENGTH (zero rows). Two kernel launches: one
 * pass over each sequence's cache shared by all nq * g (query, head) columns,
 * then the combine of split work. */
int s4kv_multi_query_workspace_bytes(const s4kv_cache* cache, int B, int num_q_tokens, int num_q_heads,
                                     int max_seq_len, size_t* bytes);
int s4kv_multi_query_attention(s4kv_cache* cache, int layer, const void* q, int num_q_tokens,
                               int num_q_heads, const int32_t* block_table, int bt_stride,
                               const int32_t* seq_lens, const int32_t* slot_ids, int B,
                               float sm_scale, void* out, int out_dtype, void* workspace,
                               size_t ws_bytes, int max_seq_len, void* stream);

/* One decode step in one launch: appends one token to every sequence and runs
 * decode attention over the state after the append, with the result of
 * s4kv_append (one row per sequence) followed by s4kv_decode_attention.
 * Sources: "4.4 KV Cache 量化", section 3.2 (new tokens join the residual; a
 * full key group is quantized as a batch, the value leaving the window is
 * quantized; attention reads history and residual); "给 KV cache 减肥",
 * section 3.1 (compress before the write, restore when the next query reads).
 *   k_new, v_new  [B][H_kv][128] in the cache dtype: the token each sequence
 *                 appends (row b for sequence b of the call), device pointers.
 *   seq_lens      int32 [B], device: lengths AFTER this step's append (each
 *                 sequence's stored length must be seq_lens[b] - 1, else
 *                 S4KV_DEV_BAD_LENGTH; seq_lens[b] >= 1).
 *   Other arguments, the workspace rule (s4kv_decode_workspace_bytes) and the
 *   errors are those of s4kv_decode_attention; the pages and rings are left
 *   exactly as s4kv_append would leave them.
 * The kernel is a cooperative launch (every CTA resident): its CTAs append,
 * meet at a grid barrier (bounded wait: S4KV_ERR_DEVICE_TIMEOUT if it runs
 * out), then attend; a second, small launch combines split work. The barrier
 * words live in the cache's pool, so decode-step calls on one cache must not
 * overlap in time (order them on one stream). Not for the FFMA path
 * (S4KV_OPT_DECODE_IMPL = 1: S4KV_ERR_UNSUPPORTED). */
int s4kv_decode_step(s4kv_cache* cache, int layer, const void* k_new, const void* v_new, const void* q,
                     int num_q_heads, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                     const int32_t* slot_ids, int B, float sm_scale, void* out, int out_dtype, void* workspace,
                     size_t ws_bytes, int max_seq_len, void* stream);

/* Size of the device array that s4kv_decode_attention_noalloc uses as its
 * scratch: 16 MiB, held by every GPU that loads the library until exit. */
#define S4KV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Decode attention for callers that cannot allocate device memory when they
 * call it: code running while a CUDA graph is being captured, a caller whose
 * memory is fixed up front by a pool it does not own, a real-time loop that
 * must never enter the allocator. It computes exactly what
 * s4kv_decode_attention computes, with the same arguments minus the workspace:
 * the scratch is a file-scope __device__ array of S4KV_NOALLOC_SCRATCH_BYTES
 * compiled into the library. (The method's pages have no counterpart: this is
 * a packaging variant, not part of the method.)
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 *   - The first call on a device looks up the array's device address on the
 *     current device (cudaGetSymbolAddress) and keeps it; make that first call
 *     before any stream capture.
 *   - Returns S4KV_ERR_WORKSPACE_TOO_SMALL when the call would need more
 *     scratch than the array holds (s4kv_decode_workspace_bytes tells; nothing
 *     is launched then), S4KV_ERR_INVALID_ARG when the current device is not
 *     the cache's device, and S4KV_ERR_CUDA if the address lookup fails.
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (other streams, other caches, other threads) race on it and must be
 *     ordered by the caller. Nothing in the array needs to start at zero. */
int s4kv_decode_attention_noalloc(s4kv_cache* cache, int layer, const void* q, int num_q_heads,
                                  const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                                  const int32_t* slot_ids, int B, float sm_scale, void* out,
                                  int out_dtype, int max_seq_len, void* stream);

/* Restores K^, V^ of one slot exactly as attention sees them: quantized tokens
 * through fmaf(code, scale, min), residual tokens widened exactly.
 *   block_table_row int32 [>= ceil(seq_len / 16)] device pointer.
 *   out_k, out_v    fp32 [H_kv][seq_len][128] device pointers. */
int s4kv_dequant_debug(s4kv_cache* cache, int layer, int slot, const int32_t* block_table_row,
                       int seq_len, float* out_k, float* out_v, void* stream);

/* Synchronises `stream`, returns S4KV_OK, S4KV_ERR_DEVICE or
 * S4KV_ERR_DEVICE_TIMEOUT from the status word, and clears it. `detail`
 * (optional) receives the S4KV_DEV_* code. */
int s4kv_get_status(s4kv_cache* cache, void* stream, int* detail);

const char* s4kv_strerror(int status);

/* The memory ledger (no device access). */
int s4kv_kv_bytes(const s4kv_config* cfg, double batch, double tokens, s4kv_kv_bytes_report* out);

/* Tuning and test knobs.
 *   S4KV_OPT_DECODE_WARPS  largest number of worker warps of a decode call, or of
 *                          warp teams of a multi-query call (0 = all the grid
 *                          holds); fewer workers, longer slices.
 *   S4KV_OPT_DECODE_IMPL   0 = tensor-core path (mma.sync m16n8k16, default),
 *                          1 = CUDA-core FFMA path (for comparison).
 *   S4KV_OPT_TAIL_COST     weight of a tail chunk (the per-token path past the
 *                          last fully quantized group) against a key group when
 *                          the decode work is cut between warps (default 3).
 *   S4KV_OPT_WAIT_NS       limit of each bounded device wait in ns (default 1e9;
 *                          0 makes the first wait give up at once: used by the
 *                          tests of the timeout path).
 *   S4KV_OPT_MQ_KERNEL     multi-query kernel, by the call's column count nq g (0,
 *                          default) or forced. 4- and 2-bit pages: up to 48 the scales
 *                          are folded into every warp's 8 columns; from 49 each key
 *                          group is restored once and feeds tcgen05 (tensor-memory
 *                          accumulators, warp-specialized). 1 = always fold; 2 =
 *                          always restore once per team for mma.sync on 16 columns a
 *                          warp; 3 = always tcgen05.
 *                          FP8 pages: up to 48 mma.sync on 16 columns a warp, from 49
 *                          each group's codes widened once to f16 for tcgen05; 1 or 2 =
 *                          always mma.sync; 3 = always tcgen05.
 *   S4KV_OPT_KEY_SPLIT     1 (default) = decode key scores also keep the low f16
 *                          part of q' = q * scale (a second MMA per 16-channel
 *                          slice: about 22 significant bits), which keeps the
 *                          output within the tolerance when key channels are
 *                          scaled x16 or x32; 0 = f16 q' alone: about 8% faster,
 *                          but its error passes the tolerance on such channels.
 *                          Tail groups and multi-query calls always split. */
enum { S4KV_OPT_DECODE_WARPS = 1, S4KV_OPT_DECODE_IMPL = 2, S4KV_OPT_WAIT_NS = 3, S4KV_OPT_TAIL_COST = 4,
       S4KV_OPT_KEY_SPLIT = 5, S4KV_OPT_MQ_KERNEL = 6 };
int s4kv_set_option(s4kv_cache* cache, int option, long long value);

#ifdef __cplusplus
}
#endif
#endif /* S4KV_H */
