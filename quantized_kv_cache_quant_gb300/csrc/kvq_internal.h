// Launch interface between the C-ABI host layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvq {

// Quantize n_groups groups of 32 tokens per (batch row, kv head) from an fp16
// source into the grouped region, starting at group index dst_group0.
struct QuantGroupsArgs {
  const uint16_t* k_src;
  const uint16_t* v_src;
  long long src_bh_stride;  // fp16 elements between consecutive (b, h) rows of the source
  int src_tok0;             // first source token
  int n_groups;
  int dst_group0;
  int batch, kv_heads, head_dim, k_bits, v_bits, groups_cap;
  uint8_t* k_codes;
  uint8_t* k_meta;
  uint8_t* v_codes;
  uint8_t* v_meta;
};

// Copy n_tokens fp16 rows of D channels for every (b, h) (K and V together).
struct CopyTokensArgs {
  const uint16_t* k_src;
  const uint16_t* v_src;
  long long src_bh_stride;
  int src_tok0;
  uint16_t* k_dst;
  uint16_t* v_dst;
  long long dst_bh_stride;
  int dst_tok0;
  int n_tokens;
  int bh;
  int head_dim;
};
cudaError_t launch_copy_tokens(const CopyTokensArgs& a, cudaStream_t s);

// Quantize a's groups; window (optional, n_tokens > 0) is a token copy that the
// same launch makes after its groups (a prefill's window fill), or alone when
// a has no groups.
cudaError_t launch_kivi_quantize(const QuantGroupsArgs& a, cudaStream_t s, const CopyTokensArgs* window = nullptr);

// ---- paged, variable-length KIVI cache ----
// Per-sequence state travels in the kernel parameters (at most kMaxPagedSeqs
// sequences keep them under the 4 KB parameter limit), so a launch needs no
// upload and captures into a CUDA graph as it is.
constexpr int kMaxPagedSeqs = 256;

// Work ranges of one batched launch: sequence b owns items [begin[b],
// begin[b+1]) (groups for a quantize, tokens for a copy), its first source
// token is src0[b] and its first destination (group index or window row) dst0[b].
struct SeqRanges {
  int begin[kMaxPagedSeqs + 1];
  int src0[kMaxPagedSeqs];
  int dst0[kMaxPagedSeqs];
};

// Group records of a paged cache: group g of sequence b, kv head h lives in
// pool block block_table[b * groups_cap + g], entry (block * kv_heads + h) of
// the pool, its four records back to back (key codes, key meta, value codes,
// value meta).
struct PagedPools {
  const int32_t* block_table;
  int groups_cap;
  int num_blocks;
};

struct PagedQuantArgs {
  QuantGroupsArgs q;  // sources, src_bh_stride, bits and shapes; k_codes = the pool (src_tok0, n_groups,
                      // dst_group0 and the other record pointers unused)
  PagedPools pools;
  int n_seqs;
  SeqRanges r;
};
cudaError_t launch_kivi_quantize_paged(const PagedQuantArgs& a, cudaStream_t s);

struct PagedCopyArgs {
  CopyTokensArgs c;  // buffers, strides and head_dim (src_tok0, dst_tok0, n_tokens unused; bh = n_seqs * kv_heads)
  int kv_heads;
  int n_seqs;
  SeqRanges r;
};
cudaError_t launch_copy_tokens_paged(const PagedCopyArgs& a, cudaStream_t s);

struct KiviDecodeArgs {
  const uint8_t* k_codes;
  const uint8_t* k_meta;
  const uint8_t* v_codes;
  const uint8_t* v_meta;
  const uint16_t* k_res;
  const uint16_t* v_res;
  const uint16_t* q;
  int batch, kv_heads, q_heads, head_dim, k_bits, v_bits, groups_cap, res_cap;
  int n_groups, n_resid;
  // Work units of one (batch row, kv head) pair: its n_groups groups, then its
  // ceil(n_resid / 32) window chunks of kChunkUnits units each. Pair p owns
  // units [p * pair_stride, p * pair_stride + units_per_pair) of a range cut
  // into n_blocks slices of units_per_block (pair_stride > units_per_pair pads
  // every pair to whole slices); a block writes one partial per pair its slice
  // touches.
  int n_pairs;
  int units_per_pair;
  int pair_stride;
  int units_per_block;
  int n_blocks;
  int part_stride;        // partial slots per query row (>= the blocks touching one pair)
  float scale_log2;       // softmax scale * log2(e)
  float* part_o;          // [B, Hq, part_stride, D]
  float* part_ml;         // [B, Hq, part_stride, 2]
  uint32_t* counters;     // [B, H_kv] finished-split counters (zero between calls)
  uint32_t* status;
  void* out;              // [B, Hq, D]
  int out_fp32;
};
cudaError_t launch_kivi_decode(const KiviDecodeArgs& a, cudaStream_t s);
// The same decode with the tensor-core operands swapped (tokens and channels
// on the tile rows, query heads x {hi, lo} on its 8 columns), for caches whose
// kv heads serve at most kMaxGqaSwapped query heads.
constexpr int kMaxGqaSwapped = 4;
// Units one 32-token window chunk is charged in the swapped-operand decode
// (its groups cost about half the MMAs of the other kernel's, its window
// chunks about as much). Swept 6, 8, 10, 12, 16 on GB300: 8 is best (MHA 4K
// 43.3 -> 42.4 us; paged GQA-4 70.2 -> 69.9 us), 10 and above change the cut
// and cost 2-9 %.
constexpr int kTrChunkUnits = 8;
cudaError_t launch_kivi_decode_tr(const KiviDecodeArgs& a, cudaStream_t s);

// Decode over a paged cache: the pairs of sequence b (b * kv_heads + h) have
// n_groups[b] groups and n_resid[b] window tokens, U_b = n_groups[b] +
// kChunkUnits * ceil(n_resid[b] / 32) units of work each, and the ranges of
// all pairs follow one another: pair (b, h) spans pair_lead + U_b units from
// unit0[b] + h * (pair_lead + U_b), its work after the first pair_lead (a
// slice that covers only those does nothing for the pair). k_codes of the
// base arguments is the pool; k_meta, v_codes, v_meta, n_groups, n_resid,
// units_per_pair and pair_stride are unused; groups_cap is the block-table
// row length.
struct PagedSeqs {
  PagedPools pools;
  int n_seqs;
  int pair_lead;
  int unit0[kMaxPagedSeqs + 1];
  int n_groups[kMaxPagedSeqs];
  int n_resid[kMaxPagedSeqs];
};
cudaError_t launch_kivi_decode_paged(const KiviDecodeArgs& a, const PagedSeqs& seqs, cudaStream_t s);
// The swapped-operand decode over a paged cache (H_q / H_kv <= kMaxGqaSwapped).
cudaError_t launch_kivi_decode_tr_paged(const KiviDecodeArgs& a, const PagedSeqs& seqs, cudaStream_t s);


struct Fp8QuantArgs {
  const uint16_t* x;
  int batch, kv_heads, seq_len, head_dim;
  const int32_t* block_table;
  int max_blocks;
  int num_blocks;
  uint8_t* pool;
  float* scale;           // [1] or, per_head, [H_kv]
  int static_scale;
  int per_head;
  int fmt;                // 0 = E4M3, 1 = E5M2
  int value_layout;       // the in-block order: 2 keys (m16n8k32 B fragments), 1 values
  uint32_t* amax_partials;  // [per_head ? H_kv : 1][amax_blocks]
  int amax_blocks;
};
cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, cudaStream_t s);

struct Fp8DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const float* k_scale;   // [1] or, per_head, [H_kv]
  const float* v_scale;
  int per_head;
  int fmt;                // 0 = E4M3, 1 = E5M2
  const int32_t* block_table;
  const int32_t* seq_lens;
  int q_fp8;              // q.k^T on FP8 tensor cores from q8 (keys in value_layout 2)
  const uint8_t* q8;      // [B, Hq, D] E4M3 query (q_fp8)
  const float* q_scale;   // [1] (q_fp8)
  int batch, q_heads, kv_heads, head_dim, max_blocks, num_blocks;
  int splits;
  int blocks_per_split;
  float scale_log2;
  float* part_o;
  float* part_ml;
  uint32_t* counters;
  uint32_t* status;
  void* out;
  int out_fp32;
};
cudaError_t launch_fp8_decode(const Fp8DecodeArgs& a, cudaStream_t s);

// The query of one decode step in E4M3 with a per-tensor dynamic scale:
// q_scale = fl32(amax / 448) (1 when q is all zeros), then
// q8 = E4M3(fl32(q / q_scale)), row-major like q.
struct Fp8QueryArgs {
  const uint16_t* q;
  long long n;            // elements, a multiple of 8
  uint8_t* q8;
  float* q_scale;
  uint32_t* partials;     // [amax_blocks]
  int amax_blocks;
};
cudaError_t launch_fp8_quantize_query(const Fp8QueryArgs& a, cudaStream_t s);

// ---- NVFP4 paged cache ----
struct Nvfp4QuantArgs {
  const uint16_t* x;      // fp16 [B, H_kv, seq_len, D]
  int batch, kv_heads, seq_len, head_dim;
  int role;               // 0 keys, 1 values: the in-block order of the records
  const int32_t* block_table;
  int max_blocks;
  int num_blocks;
  uint8_t* pool;          // [num_blocks, H_kv, 9 * D]
  float* scale;           // [1] tensor scale
  int static_scale;
  uint32_t* amax_partials;
  int amax_blocks;
};
cudaError_t launch_nvfp4_quantize(const Nvfp4QuantArgs& a, cudaStream_t s);

struct Nvfp4DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const float* k_scale;   // [1]
  const float* v_scale;   // [1]
  const int32_t* block_table;
  const int32_t* seq_lens;
  int batch, q_heads, kv_heads, head_dim, max_blocks, num_blocks;
  int splits;
  int blocks_per_split;
  float scale_log2;
  float* part_o;
  float* part_ml;
  uint32_t* counters;
  uint32_t* status;
  void* out;
  int out_fp32;
};
cudaError_t launch_nvfp4_decode(const Nvfp4DecodeArgs& a, cudaStream_t s);
int nvfp4_decode_blocks_per_sm(int head_dim, int gq);  // gq: query heads per kv head

// scale[0] = fl32(amax / fmax) over n_vec 16-byte vectors of fp16 at x (1 when
// all are zero): per-block amax partials, then one reducing block.
cudaError_t launch_tensor_scale(const uint16_t* x, long long n_vec, float fmax, uint32_t* partials, int blocks,
                                float* scale, cudaStream_t s);

int device_sm_count();
// Resident thread blocks per SM of the decode kernels (occupancy API, cached).
int kivi_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits);
int kivi_paged_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits);
int kivi_decode_tr_blocks_per_sm(int head_dim, int k_bits, int v_bits);
int kivi_paged_decode_tr_blocks_per_sm(int head_dim, int k_bits, int v_bits);
int fp8_decode_blocks_per_sm(int head_dim);

}  // namespace kvq
