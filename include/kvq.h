/*
 * kvq.h — quantized KV cache and decode attention over it, for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libkvq.so. Plain pointers and sizes only; every device pointer is
 * memory the caller allocated (cudaMalloc, a PyTorch tensor, a pool). The
 * library never allocates, never synchronizes and never prints: each call
 * validates its arguments on the host, enqueues kernels on `stream` (a
 * cudaStream_t passed as void*, NULL = the legacy default stream) and returns.
 * On any validation error nothing is enqueued and the cache descriptor is left
 * unchanged. Calls that work on one cache must be issued on one stream.
 *
 * Sources (the pages this library implements):
 *  [KIVI]  "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide),
 *          section 3 (grouped + residual structure, per-channel keys,
 *          per-token values, group 32, residual 128) and section 5 (FP8 E4M3).
 *  [CSDN]  "大模型量化从0到1（十三）：KV Cache 量化", section 2 (attention),
 *          section 4 (cache shape [B, H_kv, S, D]), section 5 (GQA), section 10
 *          (affine and FP8 quantization formulas, per-tensor granularity),
 *          section 13 (paged cache blocks).
 *  [YUN]   "LLM推理加速KV Cache量化压缩实战方案" (yunthe), "自定义KV Cache量化的实现
 *          路径": per-tensor FP8 scale = max|x| / 448.
 *
 * Scalar conventions: fp16 tensors are passed as uint16_t* (IEEE binary16 bit
 * patterns); all tensors are contiguous and row-major in the order given.
 * Every device buffer must start on a 256-byte boundary (KVQ_ERR_ALIGN).
 * GQA: query head hq uses kv head hq / (q_heads / kv_heads).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_NULL = 1,        /* a required pointer is NULL */
  KVQ_ERR_ARG = 2,         /* an argument is out of its documented range */
  KVQ_ERR_SHAPE = 3,       /* shapes disagree (e.g. q_heads % kv_heads != 0) */
  KVQ_ERR_CAPACITY = 4,    /* the cache or the pool cannot hold the tokens */
  KVQ_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than the size query */
  KVQ_ERR_UNSUPPORTED = 6, /* a valid but unimplemented combination */
  KVQ_ERR_CUDA = 7,        /* a kernel launch failed (cudaGetLastError) */
  KVQ_ERR_TIMEOUT = 8,     /* a device wait gave up (see the workspace status word) */
  KVQ_ERR_ALIGN = 9        /* a device buffer is not 256-byte aligned */
} kvq_status;

KVQ_API const char* kvq_status_string(kvq_status s);

/* ------------------------------------------------------------------------ */
/* KIVI 2/4-bit cache [KIVI section 3]                                       */
/* ------------------------------------------------------------------------ */

/* Shape and scheme of one layer's cache.
 *   batch, kv_heads, q_heads : B, H_kv, H_q (H_q % H_kv == 0, H_q / H_kv <= 8)
 *   head_dim                 : D, 64 or 128
 *   k_bits, v_bits           : 2 or 4
 *   group_size               : must be 32 (tokens per quantization group)
 *   residual_len             : R, 0 or a positive multiple of 32 (the newest R
 *                              tokens stay fp16; R = 0 keeps at most 31 tokens
 *                              in a 32-slot fp16 stage between flushes)
 *   max_tokens               : capacity in tokens per sequence               */
typedef struct {
  int32_t batch, kv_heads, q_heads, head_dim;
  int32_t k_bits, v_bits, group_size, residual_len, max_tokens;
} kivi_config;

/* Host-side descriptor of a cache whose six device buffers the caller owns.
 * n_grouped (a multiple of 32) and n_resid are the tokens held in the grouped
 * region and in the fp16 window; they change only through the calls below. */
typedef struct {
  kivi_config cfg;
  uint8_t* k_codes;  /* [B, H_kv, groups_cap, 32*D*k_bits/8]                 */
  uint8_t* k_meta;   /* [B, H_kv, groups_cap, 4*D]                           */
  uint8_t* v_codes;  /* [B, H_kv, groups_cap, 32*D*v_bits/8]                 */
  uint8_t* v_meta;   /* [B, H_kv, groups_cap, 128]                           */
  uint16_t* k_res;   /* fp16 [B, H_kv, res_cap, D], oldest token first      */
  uint16_t* v_res;   /* fp16 [B, H_kv, res_cap, D]                          */
  int32_t groups_cap; /* ceil(max_tokens / 32)                               */
  int32_t res_cap;    /* R, or 32 when R = 0                                 */
  int32_t n_grouped;
  int32_t n_resid;
} kivi_cache;

/* Grouped region layout (per batch row, kv head and group g of 32 tokens,
 * tokens 32g .. 32g+31). Codes, scales and zero points are those of [KIVI]
 * section 3 with the affine form of [CSDN] section 10, computed in IEEE fp32:
 *   per group of values x (keys: one channel over the 32 tokens; values: one
 *   token over its D channels): mn = min x (a zero min is stored as +0),
 *   mx = max x, s = fp16(fl32(fl32(mx - mn) / (2^b - 1))), z = mn,
 *   code = clamp(rint_even(fl32(fl32(x - z) / s)), 0, 2^b - 1), 0 if s == 0;
 *   dequantized value = code * s + z.
 * Inputs must be finite.
 *
 * Key meta (4*D bytes): D/16 x 4 records of 16 bytes, record ks*4 + tig holds
 *   fp16 {s[d0], s[d0+1], s[d0+8], s[d0+9], z[d0], z[d0+1], z[d0+8], z[d0+9]},
 *   d0 = 16*ks + 2*tig.
 * Value meta (128 bytes): 4 records of fp16 scales, then 4 of zero points;
 *   record tig holds tokens {2tig, 2tig+1, 8+2tig, 9+2tig, 16+2tig, 17+2tig,
 *   24+2tig, 25+2tig}.
 * Codes (32*D*b/8 bytes each for keys and values): 32 lanes x W 32-bit words
 *   (W = D/16 at 2 bits, D/8 at 4 bits); lane = 4*g + tig. Each word holds a
 *   pair of elements in its 16-bit halves (low half: first element):
 *     keys  : channels d0 = 16*ks + 8*r + 2*tig and d0+1 of token 8*nt + g
 *             (nt < 4, ks < D/16);
 *     values: tokens t0 = 16*ks + 8*r + 2*tig and t0+1 of channel 8*nt + g
 *             (nt < D/8, ks < 2).
 *   With NQ = 1 (keys) or D/32 (values):
 *     2 bits: word u = ks*NQ + nt/4, field f = (4*r + nt%4 + 1) mod 8 at bits [2f, 2f+2);
 *     4 bits: word u = (2*ks + r)*NQ + nt/4, field f = nt%4 at bits [4f, 4f+4).
 *   Word u of a lane is stored at 32-bit index (u/4)*128 + lane*4 + u%4.
 *   (These are the operand fragments of the mma.sync m16n8k16 tensor-core
 *   instruction, so that the decode kernel loads each lane's codes with
 *   16-byte shared-memory loads and turns them into operands with shifts and
 *   masks only.)                                                            */

/* Byte sizes of the six buffers in the order k_codes, k_meta, v_codes,
 * v_meta, k_res, v_res. */
KVQ_API kvq_status kivi_cache_sizes(const kivi_config* cfg, size_t bytes_out[6]);

/* Fill a descriptor for caller buffers bufs[6] (order as above, each at least
 * the size kivi_cache_sizes reports). The cache starts empty. No device work. */
KVQ_API kvq_status kivi_cache_init(kivi_cache* cache, const kivi_config* cfg, void* const bufs[6]);

/* Prefill [KIVI section 3.2]: start the cache from seq_len tokens.
 *   k, v : device fp16 [B, H_kv, seq_len, D]
 * With R > 0 the oldest 32*ceil(max(seq_len - R, 0)/32) tokens are quantized
 * into groups and the rest (at most R) are copied to the fp16 window; with
 * R = 0 the oldest 32*floor(seq_len/32) tokens are quantized. Any previous
 * content is discarded. KVQ_ERR_CAPACITY if seq_len > max_tokens. */
KVQ_API kvq_status kv_quant_prefill(kivi_cache* cache, const uint16_t* k, const uint16_t* v,
                            int32_t seq_len, void* stream);

/* Append one decode step's token [KIVI section 3.2]: k_new, v_new device fp16
 * [B, H_kv, D]. If the window is full (n_resid == res_cap) it is flushed first;
 * with R = 0 the 32-slot stage is flushed right after the append that fills
 * it. KVQ_ERR_CAPACITY if the cache already holds max_tokens tokens. */
KVQ_API kvq_status kv_append_token(kivi_cache* cache, const uint16_t* k_new, const uint16_t* v_new,
                           void* stream);

/* Flush [KIVI section 3.2]: quantize the oldest 32*floor(n_resid/32) window
 * tokens into groups and move the remaining n_resid % 32 tokens to the front
 * of the window. A no-op when n_resid < 32. */
KVQ_API kvq_status kv_flush_residual(kivi_cache* cache, void* stream);

/* Workspace for kv_decode_attention with this shape: a status word (uint32
 * at offset 0; kernels OR error bits into it, bit 0 = a device wait timed
 * out; it stays set until the caller clears it), one counter per (batch row,
 * head) at offset 256 that the kernels return to zero after every call, and
 * the split-K partials. Zero the whole workspace once after allocating it.
 * One workspace serves one stream: calls that overlap on the device must not
 * share it. */
KVQ_API size_t kv_decode_workspace_bytes(const kivi_config* cfg);

/* Decode attention [CSDN sections 2, 5] for one new token per sequence:
 *   out[b, hq, :] = softmax(q[b, hq, :] . K_hat^T * softmax_scale) V_hat
 * over the grouped tokens followed by the window tokens of kv head
 * hq / (H_q/H_kv), where K_hat, V_hat are the dequantized values.
 *   q   : device fp16 [B, H_q, D]
 *   out : device [B, H_q, D], fp32 if out_fp32 != 0, else fp16
 *   softmax_scale <= 0 selects 1/sqrt(D)
 *   ws  : workspace of at least kv_decode_workspace_bytes(cfg) bytes
 * Split-K ("flash-decoding"), one kernel launch: token chunks of each
 * (b, kv head) go to separate thread blocks, each writes (m, l, o) partials,
 * and the last block of that (b, kv head) to finish merges them with a
 * log-sum-exp reduction. Dequantization happens in registers.
 * KVQ_ERR_ARG if the cache is empty. */
KVQ_API kvq_status kv_decode_attention(const kivi_cache* cache, const uint16_t* q, void* out,
                               int32_t out_fp32, float softmax_scale, void* ws,
                               size_t ws_bytes, void* stream);

/* Decode attention for callers that cannot allocate device memory. The pages
 * describe nothing like it; it exists for users of this library. Some callers
 * may not call cudaMalloc: for example a serving engine that has handed all
 * free device memory to a fixed KV-block pool before it starts stepping, or a
 * plugin whose host framework forbids allocation while a step runs. This call
 * computes exactly what kv_decode_attention computes (same kernel, same
 * arguments minus the workspace) but keeps its split-K scratch in one
 * file-scope device array of KVQ_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU
 * loading the library holds until the process exits; it allocates nothing.
 *   - The scratch a call needs is 256 + 4*B*H_q (rounded up to 256) +
 *     4*B*H_q*S*(D+2) bytes, S the number of token splits the call picks
 *     (at most 64); a call that would need more returns KVQ_ERR_CAPACITY and
 *     enqueues nothing.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and zeroes the array's status word; make that
 *     first call before any stream capture. The address is kept for the life
 *     of the process: calling this after cudaDeviceReset in the same process
 *     is not supported (the reset unloads the array).
 *   - Every call shares the one array and clears its split counters with an
 *     asynchronous memset on `stream` first. Calls that overlap on the GPU
 *     (other streams, other host threads) race on it: serialize them.
 *   - Like the workspace status word of kv_decode_attention, the array's
 *     status word collects the error bits of every call (bit 0 = a device
 *     wait timed out) until kv_decode_noalloc_status clears it. */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
KVQ_API kvq_status kv_decode_attention_noalloc(const kivi_cache* cache, const uint16_t* q, void* out,
                                               int32_t out_fp32, float softmax_scale, void* stream);

/* Reads the status word of kv_decode_attention_noalloc's scratch array on the
 * current device into *status (host memory): it enqueues the copy on `stream`
 * and waits for that stream, so the word covers every call enqueued on it
 * before. With clear != 0 the word is then zeroed (enqueued on `stream`).
 * Returns KVQ_ERR_TIMEOUT when bit 0 is set, else KVQ_OK. Not for use during
 * stream capture. */
KVQ_API kvq_status kv_decode_noalloc_status(uint32_t* status, int32_t clear, void* stream);

/* ------------------------------------------------------------------------ */
/* Paged, variable-length KIVI cache [KIVI section 3, CSDN section 13]       */
/* ------------------------------------------------------------------------ */

/* A batch of sequences of different lengths. Each sequence is a KIVI cache of
 * its own (the rules above: prefill split, window, flush timing, all on the
 * sequence's own length); its groups of 32 tokens live in blocks of one shared
 * pool, reached through a block table as in [CSDN] section 13. The pages
 * combine the two ideas without fixing a layout; this one is the library's:
 * one pool block holds one group of one sequence for every kv head, and for
 * each kv head the four records of the contiguous cache (same byte layout per
 * record) back to back, so that one group of one head is one contiguous run.
 *
 *   pool    : [num_blocks, H_kv, E] bytes, E = KC + KM + VC + 128 with
 *             KC = 32*D*k_bits/8 (key codes at offset 0), KM = 4*D (key meta
 *             at KC), VC = 32*D*v_bits/8 (value codes at KC + KM), value meta
 *             at KC + KM + VC
 *   windows : fp16 k_res, v_res [B, H_kv, res_cap, D], one per sequence
 *   table   : device int32 block_table [B, groups_cap], groups_cap =
 *             ceil(max_tokens / 32); entry [b, g] is the pool block of group g
 *             of sequence b. The caller owns and fills it (the block
 *             allocator is the caller's): every group a call writes or reads
 *             needs an entry in [0, num_blocks), and two groups held at the
 *             same time need different blocks. A quantize skips a group whose
 *             entry is outside [0, num_blocks) (nothing is written); the decode
 *             clamps such entries into the pool (wrong numbers, no access
 *             outside it).
 * Sequence b's state is n_grouped[b] (a multiple of 32) and n_resid[b], kept
 * on the host in the descriptor. Groups written by a call: prefill, groups 0
 * .. n_grouped[b]/32 - 1 after it; append, when n_resid[b] == res_cap before
 * it (R > 0), groups n_grouped[b]/32 .. + R/32 - 1, and with R = 0, when
 * n_resid[b] == 31, group n_grouped[b]/32; flush, groups n_grouped[b]/32 ..
 * + floor(n_resid[b]/32) - 1. */
#define KVQ_PAGED_MAX_SEQS 256

/* cfg.batch is the number of sequences (1 .. KVQ_PAGED_MAX_SEQS), cfg.max_tokens
 * the capacity of one sequence; num_blocks >= 1 is the pool size in blocks. */
typedef struct {
  kivi_config cfg;
  int32_t num_blocks;
} kivi_paged_config;

typedef struct {
  kivi_paged_config pcfg;
  uint8_t* pool;
  uint16_t* k_res;
  uint16_t* v_res;
  const int32_t* block_table;
  int32_t groups_cap;  /* block-table row length, ceil(max_tokens / 32)       */
  int32_t res_cap;     /* R, or 32 when R = 0                                 */
  int32_t n_grouped[KVQ_PAGED_MAX_SEQS];
  int32_t n_resid[KVQ_PAGED_MAX_SEQS];
} kivi_paged_cache;

/* Byte sizes of the three buffers: the pool, then the k_res and v_res windows. */
KVQ_API kvq_status kivi_paged_cache_sizes(const kivi_paged_config* cfg, size_t bytes_out[3]);

/* Fill a descriptor for caller buffers bufs[3] and the caller's block table
 * (device int32 [B, groups_cap]). Every sequence starts empty. No device work.
 * KVQ_ERR_UNSUPPORTED for more than KVQ_PAGED_MAX_SEQS sequences. */
KVQ_API kvq_status kivi_paged_cache_init(kivi_paged_cache* cache, const kivi_paged_config* cfg,
                                         void* const bufs[3], const int32_t* block_table);

/* Prefill every sequence: sequence b starts from its first seq_lens[b] tokens
 * of k, v (device fp16 [B, H_kv, max_seq_len, D]); seq_lens is a HOST int32
 * array of B entries in [0, max_seq_len]. Each sequence is split as
 * kv_quant_prefill splits one cache (0 tokens leave it empty); one quantize
 * and one copy launch serve all sequences. Previous content is discarded.
 * KVQ_ERR_CAPACITY if some seq_lens[b] > max_tokens. */
KVQ_API kvq_status kv_paged_prefill(kivi_paged_cache* cache, const uint16_t* k, const uint16_t* v,
                                    int32_t max_seq_len, const int32_t* seq_lens, void* stream);

/* Append one token to every sequence: k_new, v_new device fp16 [B, H_kv, D].
 * Each sequence flushes as kv_append_token does (full windows are flushed
 * before the copy, a full 32-slot stage right after it when R = 0), batched
 * into one quantize launch. KVQ_ERR_CAPACITY if some sequence already holds
 * max_tokens tokens. */
KVQ_API kvq_status kv_paged_append(kivi_paged_cache* cache, const uint16_t* k_new, const uint16_t* v_new,
                                   void* stream);

/* Flush every sequence as kv_flush_residual flushes one cache. */
KVQ_API kvq_status kv_paged_flush(kivi_paged_cache* cache, void* stream);

/* Workspace of kv_paged_decode_attention (the layout and rules of
 * kv_decode_workspace_bytes, B = the number of sequences). */
KVQ_API size_t kv_paged_decode_workspace_bytes(const kivi_paged_config* cfg);

/* Decode attention of one new token per sequence, as kv_decode_attention,
 * over sequence b's own grouped tokens then window tokens. q: device fp16
 * [B, H_q, D]; out: device [B, H_q, D] (fp32 if out_fp32). The work of all
 * (sequence, kv head) pairs is cut into equal slices of one launch whatever
 * the lengths (split-K across pairs, one partial per pair a slice touches,
 * log-sum-exp merge by the last slice of each pair). KVQ_ERR_ARG if some
 * sequence is empty; KVQ_ERR_UNSUPPORTED if the work of all pairs exceeds
 * 2^31 units (one unit per group, about 6 per 32 window tokens). */
KVQ_API kvq_status kv_paged_decode_attention(const kivi_paged_cache* cache, const uint16_t* q, void* out,
                                             int32_t out_fp32, float softmax_scale, void* ws,
                                             size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 paged cache [KIVI section 5, CSDN section 10, YUN]               */
/* ------------------------------------------------------------------------ */

/* Roles of a paged pool: the library fixes each role's in-block byte order;
 * the decode calls take one pool of each and refuse them swapped. */
#define KVQ_ROLE_KEY 0
#define KVQ_ROLE_VALUE 1

/* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest finite 448.
 * Encoding rounds to nearest even; magnitudes >= 448 (and infinities)
 * saturate to +-448; NaN encodes as 0x7F. E5M2 ([CSDN] section 18.4): 1 sign,
 * 5 exponent bits (bias 15), 2 mantissa bits; largest finite 57344; round to
 * nearest even, saturating to +-57344, NaN -> 0x7F.
 *
 * Pool layout: pool[num_blocks, H_kv, 16 * D] bytes; logical token t of
 * sequence b lives in physical block block_table[b * max_blocks + t/16], row
 * t % 16 ([CSDN] section 13). Within one (block, kv head) the 16*D bytes are
 * stored in tensor-core fragment order (lane = 4*g + tig, D/2 bytes per lane;
 * byte p of lane l's stream is stored at byte ((p/16)*32 + l)*16 + p%16):
 *   KVQ_ROLE_KEY   : 4-byte word w = (nt*(D/32) + kk)*2 + r of a lane holds
 *                    channels 32*kk + 16*r + 4*tig .. +3 of token 8*nt + g
 *                    (nt < 2): the B fragments of mma.sync m16n8k32 (FP8
 *                    operands), and, with the query's channels permuted
 *                    alike, those of m16n8k16 after an exact fp16 conversion;
 *   KVQ_ROLE_VALUE : byte pair i = nt*2 + r of a lane holds tokens
 *                    t0 = 8*r + 2*tig, t0+1 of channel 8*nt + g (nt < D/8).
 * Rows of a block past the end of the sequence are written as zero bytes. */

/* Host-side descriptor of one FP8 pool (device memory owned by the caller). */
typedef struct {
  int32_t role;        /* KVQ_ROLE_KEY or KVQ_ROLE_VALUE: fixes the in-block order */
  int32_t fp8_format;  /* 0 = E4M3 (FMAX 448), 1 = E5M2 (FMAX 57344)                */
  int32_t per_head;    /* 0: one scale for the tensor; 1: one per kv head [CSDN 10.1] */
  int32_t num_blocks;
  int32_t kv_heads;
  int32_t head_dim;    /* 64 or 128 */
  uint8_t* pool;       /* device [num_blocks, kv_heads, 16 * head_dim]              */
  float* scale;        /* device float32 [1] (per_head == 0) or [kv_heads]           */
} fp8_pool;

/* Bytes of the pool buffer for this shape (0 if the shape is invalid). */
KVQ_API size_t fp8_pool_bytes(int32_t num_blocks, int32_t kv_heads, int32_t head_dim);

/* Fill a descriptor; no device work. KVQ_ERR_ARG for a role, fp8_format or
 * per_head out of range or num_blocks, kv_heads <= 0; KVQ_ERR_UNSUPPORTED for
 * head_dim other than 64, 128. */
KVQ_API kvq_status fp8_pool_init(fp8_pool* pool, int32_t role, int32_t fp8_format, int32_t per_head,
                                 int32_t num_blocks, int32_t kv_heads, int32_t head_dim, void* buf, float* scale);

/* Workspace of fp8_kv_quantize: per-block amax partials (4096 words, for one
 * scale or split between the per-head scales). */
KVQ_API size_t fp8_quantize_workspace_bytes(int32_t batch, int32_t kv_heads, int32_t seq_len, int32_t head_dim);

/* Quantize one tensor (K or V, as the pool's role says) of one layer into the pool.
 *   x           : device fp16 [B, kv_heads, seq_len, D]
 *   block_table : device int32 [B, max_blocks]; blocks whose entry lies
 *                 outside [0, num_blocks) are skipped (nothing written)
 *   static_scale: 0: the pool's scale is written with fl32(amax/FMAX), amax =
 *                 max|x| over the whole tensor (or over kv head h's slice for
 *                 scale[h]), scale 1 where amax == 0 [YUN]; 1: the scale is
 *                 read as given (e.g. 1.0, the no-calibration route of [KIVI]
 *                 section 6.1).
 * byte = FP8(fl32(x / scale)). KVQ_ERR_CAPACITY if ceil(seq_len/16) > max_blocks. */
KVQ_API kvq_status fp8_kv_quantize(const fp8_pool* pool, const uint16_t* x, int32_t batch, int32_t seq_len,
                                   const int32_t* block_table, int32_t max_blocks, int32_t static_scale, void* ws,
                                   size_t ws_bytes, void* stream);

/* Workspace of fp8_decode_attention: the layout of kv_decode_workspace_bytes
 * (status word, split counters, partials) for this batch and q_heads, then, at
 * byte offset kv_decode_workspace_bytes of the same shape, the E4M3 query of
 * a q_fp8 call (B*H_q*D bytes, row-major like q, the region rounded up to 256
 * bytes), its float32 scale (one value in a 256-byte slot) and 1 KiB of amax
 * partials. */
KVQ_API size_t fp8_decode_workspace_bytes(int32_t batch, int32_t q_heads, int32_t head_dim);

/* Decode attention over the FP8 paged cache:
 *   out[b, hq] = softmax(q . (k_scale * K)^T * softmax_scale) (v_scale * V)
 * over tokens 0 .. seq_lens[b]-1 of kv head hq / (H_q/H_kv).
 *   k, v     : a KVQ_ROLE_KEY and a KVQ_ROLE_VALUE pool of the same shape,
 *              format and scale granularity (KVQ_ERR_ARG for swapped roles or
 *              different formats or granularities, KVQ_ERR_SHAPE for shapes)
 *   q        : device fp16 [B, H_q, D];  out: device [B, H_q, D] (fp32 or fp16)
 *   q_fp8    : 0: q stays fp16 (scores from q and the exactly converted keys);
 *              1: FP8-domain attention ([CSDN] section 18.7: with FP8 KV and
 *              FlashAttention-3 the query is quantized too): q is quantized to
 *              E4M3 with the per-tensor dynamic scale q_scale = fl32(amax_q /
 *              448) over the whole q (1 if q is all zeros), byte =
 *              E4M3(fl32(q / q_scale)), and the scores are (E4M3 q) . (FP8 k)
 *              * q_scale * k_scale on FP8 tensor cores. The softmax weights
 *              stay fp32 for p.V.
 *   seq_lens : device int32 [B], each in [1, max_seq_len]
 * The host passes max_seq_len >= every seq_lens[b] (it sizes the grid) and
 * max_seq_len <= max_blocks*16. Block-table entries must lie in
 * [0, num_blocks); the kernels clamp them (and seq_lens) so that a bad table
 * gives wrong numbers but never an access outside the pool or the table. */
KVQ_API kvq_status fp8_decode_attention(const uint16_t* q, const fp8_pool* k, const fp8_pool* v, int32_t q_fp8,
                                        const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                        int32_t q_heads, int32_t max_blocks, int32_t max_seq_len, void* out,
                                        int32_t out_fp32, float softmax_scale, void* ws, size_t ws_bytes,
                                        void* stream);

/* ------------------------------------------------------------------------ */
/* NVFP4 paged cache [CSDN sections 21.2, 21.3, 13]                          */
/* ------------------------------------------------------------------------ */

/* [CSDN] section 21.2 names NVFP4 KV as the more aggressive 4-bit
 * floating-point cache path of Blackwell-class GPUs (about 1/4 of the BF16
 * bytes, section 21.3) without giving its format. This library follows
 * NVIDIA's public NVFP4 definition, with the tensor scale from the pages'
 * per-tensor amax rule:
 *   element : E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit;
 *             magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), round to nearest even,
 *             saturating to +-6. Inputs must be finite.
 *   block   : 16 consecutive channels of one token share one E4M3 scale byte
 *             b = E4M3(fl32(fl32(amax_b / 6) / s_t)), S_b = e4m3(b).
 *   tensor  : one float32 scale s_t per tensor (K or V of a layer):
 *             dynamic s_t = fl32(amax / 2688) (2688 = 448 * 6; 1 for an
 *             all-zero tensor), or a static (calibrated) value.
 *   code    = E2M1(fl32(x / fl32(S_b * s_t))), 0 for the whole block when
 *             S_b = 0; dequantized value = e2m1(code) * S_b * s_t.
 *
 * Pool: [num_blocks, kv_heads, 9*D] bytes; one (block, kv head) record holds
 * 16 tokens: 8*D bytes of codes, then D scale bytes. Logical token t of
 * sequence b lives in block block_table[b * max_blocks + t/16], row t % 16.
 * Within a record (lane = 4*g + tig; byte p of a lane's code stream at byte
 * ((p/16)*32 + lane)*16 + p%16 of the record):
 *   KVQ_ROLE_KEY   : code byte i = (nt*(D/16) + ks)*2 + r of a lane holds
 *                    channels c0 = 16*ks + 8*r + 2*tig (low nibble) and c0+1
 *                    (high nibble) of token 8*nt + g (nt < 2); scale byte
 *                    g*(D/8) + nt*(D/16) + ks is the scale of token 8*nt + g,
 *                    channels 16*ks .. 16*ks + 15;
 *   KVQ_ROLE_VALUE : code byte i = nt*2 + r holds tokens t0 = 8*r + 2*tig (low
 *                    nibble) and t0+1 (high nibble) of channel 8*nt + g
 *                    (nt < D/8); scale byte ((tig*2 + r)*(D/16) + j)*2 + e is
 *                    the scale of token 8*r + 2*tig + e, channels 16*j .. +15.
 * (These are the m16n8k16 operand fragments of q.k^T and p.V, with each
 * lane's block scales next to each other.) Rows past the end of a sequence
 * hold zero codes and zero scales. */
/* Host-side descriptor of one NVFP4 pool (device memory owned by the caller). */
typedef struct {
  int32_t role;        /* KVQ_ROLE_KEY or KVQ_ROLE_VALUE: fixes the in-block order */
  int32_t num_blocks;
  int32_t kv_heads;
  int32_t head_dim;    /* 64 or 128 */
  uint8_t* pool;       /* device [num_blocks, kv_heads, 9 * head_dim] */
  float* tensor_scale; /* device float32 [1] */
} nvfp4_pool;

/* Bytes of the pool buffer for this shape (0 if the shape is invalid). */
KVQ_API size_t nvfp4_pool_bytes(int32_t num_blocks, int32_t kv_heads, int32_t head_dim);

/* Fill a descriptor; no device work. KVQ_ERR_ARG for a role other than
 * KVQ_ROLE_KEY / KVQ_ROLE_VALUE or num_blocks, kv_heads <= 0;
 * KVQ_ERR_UNSUPPORTED for head_dim other than 64, 128. */
KVQ_API kvq_status nvfp4_pool_init(nvfp4_pool* pool, int32_t role, int32_t num_blocks, int32_t kv_heads,
                                   int32_t head_dim, void* buf, float* tensor_scale);

/* Workspace of nvfp4_kv_quantize with a dynamic scale (amax partials). */
KVQ_API size_t nvfp4_quantize_workspace_bytes(void);

/* Quantize one tensor (K or V, as the pool's role says) into the pool.
 *   x           : device fp16 [B, kv_heads, seq_len, D]
 *   block_table : device int32 [B, max_blocks]; blocks whose entry lies
 *                 outside [0, num_blocks) are skipped (nothing written)
 *   static_scale: 0 = write the dynamic s_t to *tensor_scale first; 1 = read
 *                 *tensor_scale as given (a calibrated scale, > 0)
 *   ws          : nvfp4_quantize_workspace_bytes() bytes when static_scale == 0
 * KVQ_ERR_CAPACITY if ceil(seq_len/16) > max_blocks. */
KVQ_API kvq_status nvfp4_kv_quantize(const nvfp4_pool* pool, const uint16_t* x, int32_t batch, int32_t seq_len,
                                     const int32_t* block_table, int32_t max_blocks, int32_t static_scale, void* ws,
                                     size_t ws_bytes, void* stream);

/* Workspace of nvfp4_decode_attention (the layout of kv_decode_workspace_bytes). */
KVQ_API size_t nvfp4_decode_workspace_bytes(int32_t batch, int32_t q_heads, int32_t head_dim);

/* Decode attention over the NVFP4 paged cache:
 *   out[b, hq] = softmax(q . K_hat^T * softmax_scale) V_hat
 * over tokens 0 .. seq_lens[b]-1 of kv head hq / (H_q/H_kv), with K_hat and
 * V_hat the dequantized values of the two pools.
 *   k, v     : descriptors of a KVQ_ROLE_KEY and a KVQ_ROLE_VALUE pool of the
 *              same shape (KVQ_ERR_ARG otherwise)
 *   q        : device fp16 [B, H_q, D];  out: device [B, H_q, D] (fp32 or fp16)
 *   seq_lens : device int32 [B], each in [1, max_seq_len]; max_seq_len <=
 *              max_blocks*16 (the host sizes the grid from it)
 * Split-K over the blocks of each sequence, merged by the last block of each
 * (b, kv head) as in fp8_decode_attention. Table entries and seq_lens are
 * clamped on the device: a bad table gives wrong numbers, never an access
 * outside the pool. */
KVQ_API kvq_status nvfp4_decode_attention(const uint16_t* q, const nvfp4_pool* k, const nvfp4_pool* v,
                                          const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                          int32_t q_heads, int32_t max_blocks, int32_t max_seq_len, void* out,
                                          int32_t out_fp32, float softmax_scale, void* ws, size_t ws_bytes,
                                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
