// C-ABI host layer of libkvq: argument validation, the streaming state machine
// of the KIVI cache, split-K sizing, and kernel launches. Declared in kvq.h.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_internal.h"

using kvq::kGroup;
using kvq::kMaxSplits;
using kvq::kWsHeader;

namespace {

constexpr int kAmaxBlocksMax = 4096;
constexpr int kQueryAmaxBlocks = 256;  // amax blocks over a decode query (each cast block reduces them all)
constexpr int kMinUnitsPerSplit = 8;  // groups (or paged blocks) per split: two per warp

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

kvq_status check_config(const kivi_config* c) {
  if (c == nullptr) return KVQ_ERR_NULL;
  if (c->batch <= 0 || c->kv_heads <= 0 || c->q_heads <= 0 || c->max_tokens <= 0) return KVQ_ERR_ARG;
  if (c->batch > 65535 || c->kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if ((c->k_bits != 2 && c->k_bits != 4) || (c->v_bits != 2 && c->v_bits != 4)) return KVQ_ERR_UNSUPPORTED;
  if (c->group_size != kGroup) return KVQ_ERR_UNSUPPORTED;
  if (c->residual_len < 0 || c->residual_len % kGroup != 0) return KVQ_ERR_ARG;
  if (c->q_heads % c->kv_heads != 0) return KVQ_ERR_SHAPE;
  if (c->q_heads / c->kv_heads > kvq::kMaxGqa) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

int groups_cap_of(const kivi_config* c) { return ceil_div(c->max_tokens, kGroup); }
int res_cap_of(const kivi_config* c) { return c->residual_len > 0 ? c->residual_len : kGroup; }

void record_bytes(const kivi_config* c, size_t out[6]) {
  const size_t bh = static_cast<size_t>(c->batch) * c->kv_heads;
  const size_t groups = static_cast<size_t>(groups_cap_of(c));
  const size_t d = static_cast<size_t>(c->head_dim);
  out[0] = bh * groups * (32 * d * c->k_bits / 8);
  out[1] = bh * groups * (4 * d);
  out[2] = bh * groups * (32 * d * c->v_bits / 8);
  out[3] = bh * groups * 128;
  out[4] = bh * static_cast<size_t>(res_cap_of(c)) * d * 2;
  out[5] = out[4];
}

kvq_status check_cache(const kivi_cache* cache) {
  if (cache == nullptr) return KVQ_ERR_NULL;
  const kvq_status st = check_config(&cache->cfg);
  if (st != KVQ_OK) return st;
  if (!cache->k_codes || !cache->k_meta || !cache->v_codes || !cache->v_meta || !cache->k_res || !cache->v_res)
    return KVQ_ERR_NULL;
  if (cache->groups_cap != groups_cap_of(&cache->cfg) || cache->res_cap != res_cap_of(&cache->cfg)) return KVQ_ERR_ARG;
  if (cache->n_grouped < 0 || cache->n_grouped % kGroup != 0 || cache->n_resid < 0 || cache->n_resid > cache->res_cap)
    return KVQ_ERR_ARG;
  if (cache->n_grouped + cache->n_resid > cache->cfg.max_tokens) return KVQ_ERR_ARG;
  return KVQ_OK;
}

// Quantize n whole groups from the head of the fp16 window into the grouped region.
kvq_status flush_groups(kivi_cache* c, int n_tokens, cudaStream_t s) {
  kvq::QuantGroupsArgs q{};
  q.k_src = c->k_res;
  q.v_src = c->v_res;
  q.src_bh_stride = static_cast<long long>(c->res_cap) * c->cfg.head_dim;
  q.src_tok0 = 0;
  q.n_groups = n_tokens / kGroup;
  q.dst_group0 = c->n_grouped / kGroup;
  q.batch = c->cfg.batch;
  q.kv_heads = c->cfg.kv_heads;
  q.head_dim = c->cfg.head_dim;
  q.k_bits = c->cfg.k_bits;
  q.v_bits = c->cfg.v_bits;
  q.groups_cap = c->groups_cap;
  q.k_codes = c->k_codes;
  q.k_meta = c->k_meta;
  q.v_codes = c->v_codes;
  q.v_meta = c->v_meta;
  kvq_status st = from_cuda(kvq::launch_kivi_quantize(q, s));
  if (st != KVQ_OK) return st;
  const int rest = c->n_resid - n_tokens;
  if (rest > 0) {  // rest < 32 <= n_tokens: source and destination rows do not overlap
    kvq::CopyTokensArgs m{};
    m.k_src = c->k_res;
    m.v_src = c->v_res;
    m.src_bh_stride = q.src_bh_stride;
    m.src_tok0 = n_tokens;
    m.k_dst = c->k_res;
    m.v_dst = c->v_res;
    m.dst_bh_stride = q.src_bh_stride;
    m.dst_tok0 = 0;
    m.n_tokens = rest;
    m.bh = c->cfg.batch * c->cfg.kv_heads;
    m.head_dim = c->cfg.head_dim;
    st = from_cuda(kvq::launch_copy_tokens(m, s));
    if (st != KVQ_OK) return st;
  }
  c->n_grouped += n_tokens;
  c->n_resid = rest;
  return KVQ_OK;
}

// Decode workspace: [status word | 256 B][split counters, one per (b, head) |
// rounded to 256 B][partial o: B*Hq*splits*D floats][partial (m, l)].
size_t counters_bytes(int batch, int q_heads) {
  return (static_cast<size_t>(batch) * q_heads * sizeof(uint32_t) + 255) / 256 * 256;
}

size_t decode_ws_bytes(int batch, int q_heads, int head_dim) {
  return static_cast<size_t>(kWsHeader) + counters_bytes(batch, q_heads) +
         static_cast<size_t>(batch) * q_heads * kMaxSplits * (static_cast<size_t>(head_dim) + 2) * sizeof(float);
}

// Token splits for `units` work items (groups or paged blocks) per
// (batch row, kv head), `pairs` such pairs and `extra` single-block items
// (the fp16-window blocks). Picks the split count with the smallest estimated
// time: whole waves of resident blocks times (the items one warp processes +
// a fixed per-block cost of about four items for the query set-up, the
// partial write and the merge).
int choose_splits(int units, int pairs, int max_splits, int blocks_per_sm, int extra) {
  if (units <= 0) return 0;
  const long long slots = static_cast<long long>(kvq::device_sm_count()) * std::max(1, blocks_per_sm);
  const int cap = std::max(1, std::min(max_splits, ceil_div(units, kMinUnitsPerSplit)));
  int best = 1;
  long long best_cost = LLONG_MAX;
  for (int s = 1; s <= cap; ++s) {
    const int per = ceil_div(units, s);
    const long long ctas = static_cast<long long>(pairs) * s + extra;
    const long long waves = (ctas + slots - 1) / slots;
    const long long cost = waves * (ceil_div(per, 4) + 4);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  const int per = ceil_div(units, best);
  return ceil_div(units, per);
}

// The decode grid of a KIVI cache. The work of one (batch row, kv head) pair
// is a range of units: its groups, then its fp16 window cut into 32-token
// chunks of kChunkUnits units each (a chunk is one warp's work, about two
// groups of time for the whole block). The grid holds at most as many blocks
// as the GPU keeps resident, all with the same number of units, in one of two
// cuts, whichever gives the smaller block:
//  * pair-aligned: every pair in k equal slices (no block crosses a pair), used
//    when the pairs fill the resident slots well;
//  * stream-K: the ranges of all pairs, one after the other, in equal slices; a
//    block then writes one partial per pair its slice touches and pays for
//    each extra pair about kSegmentUnits units (its pipeline drains and
//    restarts, and it may merge the pair it leaves).
struct DecodePlan {
  int n_groups;
  int units_per_pair;
  int pair_stride;
  int units_per_block;
  int n_blocks;
  int part_stride;  // the most blocks one pair can touch
};

constexpr int kSegmentUnits = 8;

// The same cost as the paged decode charges it ahead of each pair. On GB300
// (32 sequences, GQA 8, lengths 8192 each or 512 .. 16384) 8 units measured
// best: 0 leaves the blocks on short sequences behind (89.4 us against 87.2
// for the mixed lengths), 16 over-charges each pair (86.8 us against 85.0 for
// equal lengths).
constexpr int kPairLeadUnits = 8;

// The decode kernel of a contiguous cache: the swapped-operand one when a kv
// head serves at most kMaxGqaSwapped query heads (half the MMAs per group).
bool use_swapped_decode(const kivi_config& cf) { return cf.q_heads / cf.kv_heads <= kvq::kMaxGqaSwapped; }

cudaError_t launch_contiguous_decode(const kivi_config& cf, const kvq::KiviDecodeArgs& a, cudaStream_t s) {
  return use_swapped_decode(cf) ? kvq::launch_kivi_decode_tr(a, s) : kvq::launch_kivi_decode(a, s);
}

DecodePlan plan_kivi_decode(const kivi_cache* cache) {
  const kivi_config& cf = cache->cfg;
  DecodePlan p{};
  p.n_groups = cache->n_grouped / kGroup;
  const int chunk_units = use_swapped_decode(cf) ? kvq::kTrChunkUnits : kvq::kChunkUnits;
  const int U = p.n_groups + chunk_units * ceil_div(cache->n_resid, kGroup);
  p.units_per_pair = U;
  const long long pairs = static_cast<long long>(cf.batch) * cf.kv_heads;
  const int per_sm = use_swapped_decode(cf) ? kvq::kivi_decode_tr_blocks_per_sm(cf.head_dim, cf.k_bits, cf.v_bits)
                                            : kvq::kivi_decode_blocks_per_sm(cf.head_dim, cf.k_bits, cf.v_bits);
  const long long slots = static_cast<long long>(kvq::device_sm_count()) * std::max(1, per_sm);
  // stream-K slices
  long long per_s = (pairs * U + slots - 1) / slots;
  per_s = std::max<long long>(per_s, kMinUnitsPerSplit);
  per_s = std::max<long long>(per_s, ceil_div(U, kMaxSplits - 1));  // <= kMaxSplits partials per pair
  const long long extra_pairs = (per_s - 1) / U + 1;                 // pairs a slice can touch, minus one
  const long long cost_s = per_s + kSegmentUnits * extra_pairs;
  // pair-aligned slices
  if (pairs <= slots) {
    int k = static_cast<int>(slots / pairs);
    k = std::min(k, std::max(1, ceil_div(U, kMinUnitsPerSplit)));
    k = std::min(k, kMaxSplits);
    const int per_a = ceil_div(U, k);
    k = ceil_div(U, per_a);  // no empty slice
    if (per_a <= cost_s) {
      p.units_per_block = per_a;
      p.pair_stride = k * per_a;
      p.n_blocks = static_cast<int>(pairs * k);
      p.part_stride = k;
      return p;
    }
  }
  p.units_per_block = static_cast<int>(per_s);
  p.pair_stride = U;
  p.n_blocks = static_cast<int>((pairs * U + per_s - 1) / per_s);
  p.part_stride = std::min(kMaxSplits, ceil_div(U, p.units_per_block) + 1);
  return p;
}

kvq::KiviDecodeArgs kivi_decode_args(const kivi_cache* cache, const DecodePlan& plan, const uint16_t* q, void* out,
                                     int32_t out_fp32, float scale, uint8_t* ws) {
  const kivi_config& cf = cache->cfg;
  kvq::KiviDecodeArgs a{};
  a.k_codes = cache->k_codes;
  a.k_meta = cache->k_meta;
  a.v_codes = cache->v_codes;
  a.v_meta = cache->v_meta;
  a.k_res = cache->k_res;
  a.v_res = cache->v_res;
  a.q = q;
  a.batch = cf.batch;
  a.kv_heads = cf.kv_heads;
  a.q_heads = cf.q_heads;
  a.head_dim = cf.head_dim;
  a.k_bits = cf.k_bits;
  a.v_bits = cf.v_bits;
  a.groups_cap = cache->groups_cap;
  a.res_cap = cache->res_cap;
  a.n_groups = plan.n_groups;
  a.n_resid = cache->n_resid;
  a.n_pairs = cf.batch * cf.kv_heads;
  a.units_per_pair = plan.units_per_pair;
  a.pair_stride = plan.pair_stride;
  a.units_per_block = plan.units_per_block;
  a.n_blocks = plan.n_blocks;
  a.part_stride = plan.part_stride;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.counters = reinterpret_cast<uint32_t*>(ws + kWsHeader);
  a.part_o = reinterpret_cast<float*>(ws + kWsHeader + counters_bytes(cf.batch, cf.q_heads));
  a.part_ml = a.part_o + static_cast<size_t>(cf.batch) * cf.q_heads * plan.part_stride * cf.head_dim;
  a.out = out;
  a.out_fp32 = out_fp32;
  return a;
}

// ---------------------------------------------------------------------------
// Paged, variable-length cache
// ---------------------------------------------------------------------------
kvq_status check_paged_config(const kivi_paged_config* c) {
  if (c == nullptr) return KVQ_ERR_NULL;
  const kvq_status st = check_config(&c->cfg);
  if (st != KVQ_OK) return st;
  if (c->cfg.batch > KVQ_PAGED_MAX_SEQS) return KVQ_ERR_UNSUPPORTED;
  if (c->num_blocks <= 0) return KVQ_ERR_ARG;
  return KVQ_OK;
}

void paged_record_bytes(const kivi_paged_config* pc, size_t out[3]) {
  const kivi_config* c = &pc->cfg;
  const size_t rows = static_cast<size_t>(pc->num_blocks) * c->kv_heads;
  const size_t d = static_cast<size_t>(c->head_dim);
  out[0] = rows * (32 * d * c->k_bits / 8 + 4 * d + 32 * d * c->v_bits / 8 + 128);
  out[1] = static_cast<size_t>(c->batch) * c->kv_heads * static_cast<size_t>(res_cap_of(c)) * d * 2;
  out[2] = out[1];
}

kvq_status check_paged_cache(const kivi_paged_cache* cache) {
  if (cache == nullptr) return KVQ_ERR_NULL;
  const kvq_status st = check_paged_config(&cache->pcfg);
  if (st != KVQ_OK) return st;
  if (!cache->pool || !cache->k_res || !cache->v_res || !cache->block_table) return KVQ_ERR_NULL;
  const kivi_config& cf = cache->pcfg.cfg;
  if (cache->groups_cap != groups_cap_of(&cf) || cache->res_cap != res_cap_of(&cf)) return KVQ_ERR_ARG;
  for (int b = 0; b < cf.batch; ++b) {
    const int ng = cache->n_grouped[b], nr = cache->n_resid[b];
    if (ng < 0 || ng % kGroup != 0 || nr < 0 || nr > cache->res_cap) return KVQ_ERR_ARG;
    if (static_cast<long long>(ng) + nr > cf.max_tokens) return KVQ_ERR_ARG;
    if (cf.residual_len == 0 && nr >= kGroup) return KVQ_ERR_ARG;
  }
  return KVQ_OK;
}

// One batched quantize: sequence b's counts[b] groups, read from source token
// src0[b] of its rows, written to its logical groups dst0[b] on.
kvq_status paged_quantize(const kivi_paged_cache* c, const uint16_t* k_src, const uint16_t* v_src,
                          long long src_bh_stride, const int* counts, const int* src0, const int* dst0,
                          cudaStream_t s) {
  const kivi_config& cf = c->pcfg.cfg;
  kvq::PagedQuantArgs a{};
  long long total = 0;
  for (int b = 0; b < cf.batch; ++b) {
    a.r.begin[b] = static_cast<int>(total);
    a.r.src0[b] = src0[b];
    a.r.dst0[b] = dst0[b];
    total += counts[b];
    if (total > INT_MAX) return KVQ_ERR_UNSUPPORTED;
  }
  a.r.begin[cf.batch] = static_cast<int>(total);
  if (total == 0) return KVQ_OK;
  a.q.k_src = k_src;
  a.q.v_src = v_src;
  a.q.src_bh_stride = src_bh_stride;
  a.q.batch = cf.batch;
  a.q.kv_heads = cf.kv_heads;
  a.q.head_dim = cf.head_dim;
  a.q.k_bits = cf.k_bits;
  a.q.v_bits = cf.v_bits;
  a.q.groups_cap = c->groups_cap;
  a.q.k_codes = c->pool;
  a.pools.block_table = c->block_table;
  a.pools.groups_cap = c->groups_cap;
  a.pools.num_blocks = c->pcfg.num_blocks;
  a.n_seqs = cf.batch;
  return from_cuda(kvq::launch_kivi_quantize_paged(a, s));
}

// One batched token copy into the windows: sequence b's counts[b] tokens from
// source row src0[b] to window row dst0[b].
kvq_status paged_copy(const kivi_paged_cache* c, const uint16_t* k_src, const uint16_t* v_src,
                      long long src_bh_stride, const int* counts, const int* src0, const int* dst0, cudaStream_t s) {
  const kivi_config& cf = c->pcfg.cfg;
  kvq::PagedCopyArgs a{};
  long long total = 0;
  for (int b = 0; b < cf.batch; ++b) {
    a.r.begin[b] = static_cast<int>(total);
    a.r.src0[b] = src0[b];
    a.r.dst0[b] = dst0[b];
    total += counts[b];
    if (total > INT_MAX) return KVQ_ERR_UNSUPPORTED;
  }
  a.r.begin[cf.batch] = static_cast<int>(total);
  if (total == 0) return KVQ_OK;
  a.c.k_src = k_src;
  a.c.v_src = v_src;
  a.c.src_bh_stride = src_bh_stride;
  a.c.k_dst = c->k_res;
  a.c.v_dst = c->v_res;
  a.c.dst_bh_stride = static_cast<long long>(c->res_cap) * cf.head_dim;
  a.c.bh = cf.batch * cf.kv_heads;
  a.c.head_dim = cf.head_dim;
  a.kv_heads = cf.kv_heads;
  a.n_seqs = cf.batch;
  return from_cuda(kvq::launch_copy_tokens_paged(a, s));
}

// Flush the window head of the sequences with counts[b] > 0 groups to flush:
// quantize them into groups n_grouped[b]/32 on, move what is left of the
// window (fewer than 32 tokens) to its front, and update the state.
kvq_status paged_flush_groups(kivi_paged_cache* c, const int* counts, cudaStream_t s) {
  const int B = c->pcfg.cfg.batch;
  int src0[KVQ_PAGED_MAX_SEQS], dst0[KVQ_PAGED_MAX_SEQS], rest[KVQ_PAGED_MAX_SEQS], from[KVQ_PAGED_MAX_SEQS];
  for (int b = 0; b < B; ++b) {
    src0[b] = 0;
    dst0[b] = c->n_grouped[b] / kGroup;
    from[b] = kGroup * counts[b];
    rest[b] = counts[b] > 0 ? c->n_resid[b] - from[b] : 0;  // < 32 <= from[b]: no overlap
    if (rest[b] < 0) return KVQ_ERR_ARG;
  }
  const long long win_stride = static_cast<long long>(c->res_cap) * c->pcfg.cfg.head_dim;
  kvq_status st = paged_quantize(c, c->k_res, c->v_res, win_stride, counts, src0, dst0, s);
  if (st != KVQ_OK) return st;
  for (int b = 0; b < B; ++b) dst0[b] = 0;
  st = paged_copy(c, c->k_res, c->v_res, win_stride, rest, from, dst0, s);
  if (st != KVQ_OK) return st;
  for (int b = 0; b < B; ++b) {
    if (counts[b] == 0) continue;
    c->n_grouped[b] += from[b];
    c->n_resid[b] = rest[b];
  }
  return KVQ_OK;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_NULL: return "a required pointer is NULL";
    case KVQ_ERR_ARG: return "an argument is out of range";
    case KVQ_ERR_SHAPE: return "shapes disagree";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_UNSUPPORTED: return "unsupported combination";
    case KVQ_ERR_CUDA: return "CUDA launch failed";
    case KVQ_ERR_TIMEOUT: return "a device wait timed out";
    case KVQ_ERR_ALIGN: return "a device buffer is not 256-byte aligned";
  }
  return "unknown status";
}

kvq_status kivi_cache_sizes(const kivi_config* cfg, size_t bytes_out[6]) {
  const kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  if (bytes_out == nullptr) return KVQ_ERR_NULL;
  record_bytes(cfg, bytes_out);
  return KVQ_OK;
}

kvq_status kivi_cache_init(kivi_cache* cache, const kivi_config* cfg, void* const bufs[6]) {
  if (cache == nullptr || bufs == nullptr) return KVQ_ERR_NULL;
  const kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  for (int i = 0; i < 6; ++i) {
    if (bufs[i] == nullptr) return KVQ_ERR_NULL;
    if (!aligned(bufs[i])) return KVQ_ERR_ALIGN;
  }
  kivi_cache c{};
  c.cfg = *cfg;
  c.k_codes = static_cast<uint8_t*>(bufs[0]);
  c.k_meta = static_cast<uint8_t*>(bufs[1]);
  c.v_codes = static_cast<uint8_t*>(bufs[2]);
  c.v_meta = static_cast<uint8_t*>(bufs[3]);
  c.k_res = static_cast<uint16_t*>(bufs[4]);
  c.v_res = static_cast<uint16_t*>(bufs[5]);
  c.groups_cap = groups_cap_of(cfg);
  c.res_cap = res_cap_of(cfg);
  c.n_grouped = 0;
  c.n_resid = 0;
  *cache = c;
  return KVQ_OK;
}

kvq_status kv_quant_prefill(kivi_cache* cache, const uint16_t* k, const uint16_t* v, int32_t seq_len, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (seq_len < 0) return KVQ_ERR_ARG;
  if (seq_len > cache->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  if (seq_len > 0 && (k == nullptr || v == nullptr)) return KVQ_ERR_NULL;
  if (seq_len > 0 && (!aligned(k) || !aligned(v))) return KVQ_ERR_ALIGN;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = cache->cfg.residual_len;
  const int grouped = (R > 0) ? kGroup * ceil_div(std::max(seq_len - R, 0), kGroup) : kGroup * (seq_len / kGroup);
  const int resid = seq_len - grouped;
  kivi_cache c = *cache;
  // the window fill: tokens [grouped, seq_len) of every (b, h) to rows 0.. of the window
  kvq::CopyTokensArgs m{};
  if (resid > 0) {
    m.k_src = k;
    m.v_src = v;
    m.src_bh_stride = static_cast<long long>(seq_len) * c.cfg.head_dim;
    m.src_tok0 = grouped;
    m.k_dst = c.k_res;
    m.v_dst = c.v_res;
    m.dst_bh_stride = static_cast<long long>(c.res_cap) * c.cfg.head_dim;
    m.dst_tok0 = 0;
    m.n_tokens = resid;
    m.bh = c.cfg.batch * c.cfg.kv_heads;
    m.head_dim = c.cfg.head_dim;
  }
  {
    // one launch: the groups, then (same grid, as blocks run out of groups) the window fill
    kvq::QuantGroupsArgs q{};
    q.k_src = k;
    q.v_src = v;
    q.src_bh_stride = static_cast<long long>(seq_len) * c.cfg.head_dim;
    q.src_tok0 = 0;
    q.n_groups = grouped / kGroup;
    q.dst_group0 = 0;
    q.batch = c.cfg.batch;
    q.kv_heads = c.cfg.kv_heads;
    q.head_dim = c.cfg.head_dim;
    q.k_bits = c.cfg.k_bits;
    q.v_bits = c.cfg.v_bits;
    q.groups_cap = c.groups_cap;
    q.k_codes = c.k_codes;
    q.k_meta = c.k_meta;
    q.v_codes = c.v_codes;
    q.v_meta = c.v_meta;
    st = from_cuda(kvq::launch_kivi_quantize(q, s, &m));
    if (st != KVQ_OK) return st;
  }
  cache->n_grouped = grouped;
  cache->n_resid = resid;
  return KVQ_OK;
}

kvq_status kv_append_token(kivi_cache* cache, const uint16_t* k_new, const uint16_t* v_new, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_NULL;
  if (!aligned(k_new) || !aligned(v_new)) return KVQ_ERR_ALIGN;
  if (cache->n_grouped + cache->n_resid + 1 > cache->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  kivi_cache c = *cache;
  if (c.n_resid == c.res_cap) {
    st = flush_groups(&c, c.res_cap, s);
    if (st != KVQ_OK) return st;
  }
  kvq::CopyTokensArgs m{};
  m.k_src = k_new;
  m.v_src = v_new;
  m.src_bh_stride = c.cfg.head_dim;
  m.src_tok0 = 0;
  m.k_dst = c.k_res;
  m.v_dst = c.v_res;
  m.dst_bh_stride = static_cast<long long>(c.res_cap) * c.cfg.head_dim;
  m.dst_tok0 = c.n_resid;
  m.n_tokens = 1;
  m.bh = c.cfg.batch * c.cfg.kv_heads;
  m.head_dim = c.cfg.head_dim;
  st = from_cuda(kvq::launch_copy_tokens(m, s));
  if (st != KVQ_OK) return st;
  c.n_resid += 1;
  if (c.cfg.residual_len == 0 && c.n_resid == kGroup) {
    st = flush_groups(&c, kGroup, s);
    if (st != KVQ_OK) return st;
  }
  *cache = c;
  return KVQ_OK;
}

kvq_status kv_flush_residual(kivi_cache* cache, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  const int n = kGroup * (cache->n_resid / kGroup);
  if (n == 0) return KVQ_OK;
  kivi_cache c = *cache;
  st = flush_groups(&c, n, static_cast<cudaStream_t>(stream));
  if (st != KVQ_OK) return st;
  *cache = c;
  return KVQ_OK;
}

size_t kv_decode_workspace_bytes(const kivi_config* cfg) {
  if (check_config(cfg) != KVQ_OK) return 0;
  return decode_ws_bytes(cfg->batch, cfg->q_heads, cfg->head_dim);
}

kvq_status kv_decode_attention(const kivi_cache* cache, const uint16_t* q, void* out, int32_t out_fp32,
                               float softmax_scale, void* ws, size_t ws_bytes, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (q == nullptr || out == nullptr) return KVQ_ERR_NULL;
  if (!aligned(q) || !aligned(out)) return KVQ_ERR_ALIGN;
  if (ws == nullptr) return KVQ_ERR_WORKSPACE;
  if (!aligned(ws)) return KVQ_ERR_ALIGN;
  const kivi_config& cf = cache->cfg;
  if (ws_bytes < decode_ws_bytes(cf.batch, cf.q_heads, cf.head_dim)) return KVQ_ERR_WORKSPACE;
  if (cache->n_grouped + cache->n_resid == 0) return KVQ_ERR_ARG;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return KVQ_ERR_ARG;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cf.head_dim));

  const DecodePlan plan = plan_kivi_decode(cache);
  const kvq::KiviDecodeArgs a = kivi_decode_args(cache, plan, q, out, out_fp32, scale, static_cast<uint8_t*>(ws));
  return from_cuda(launch_contiguous_decode(cf, a, static_cast<cudaStream_t>(stream)));
}

kvq_status kivi_paged_cache_sizes(const kivi_paged_config* cfg, size_t bytes_out[3]) {
  const kvq_status st = check_paged_config(cfg);
  if (st != KVQ_OK) return st;
  if (bytes_out == nullptr) return KVQ_ERR_NULL;
  paged_record_bytes(cfg, bytes_out);
  return KVQ_OK;
}

kvq_status kivi_paged_cache_init(kivi_paged_cache* cache, const kivi_paged_config* cfg, void* const bufs[3],
                                 const int32_t* block_table) {
  if (cache == nullptr || bufs == nullptr || block_table == nullptr) return KVQ_ERR_NULL;
  const kvq_status st = check_paged_config(cfg);
  if (st != KVQ_OK) return st;
  for (int i = 0; i < 3; ++i) {
    if (bufs[i] == nullptr) return KVQ_ERR_NULL;
    if (!aligned(bufs[i])) return KVQ_ERR_ALIGN;
  }
  if (!aligned(block_table)) return KVQ_ERR_ALIGN;
  kivi_paged_cache c{};
  c.pcfg = *cfg;
  c.pool = static_cast<uint8_t*>(bufs[0]);
  c.k_res = static_cast<uint16_t*>(bufs[1]);
  c.v_res = static_cast<uint16_t*>(bufs[2]);
  c.block_table = block_table;
  c.groups_cap = groups_cap_of(&cfg->cfg);
  c.res_cap = res_cap_of(&cfg->cfg);
  *cache = c;
  return KVQ_OK;
}

kvq_status kv_paged_prefill(kivi_paged_cache* cache, const uint16_t* k, const uint16_t* v, int32_t max_seq_len,
                            const int32_t* seq_lens, void* stream) {
  kvq_status st = check_paged_cache(cache);
  if (st != KVQ_OK) return st;
  if (seq_lens == nullptr) return KVQ_ERR_NULL;
  if (max_seq_len < 0) return KVQ_ERR_ARG;
  const kivi_config& cf = cache->pcfg.cfg;
  const int B = cf.batch, R = cf.residual_len;
  int groups[KVQ_PAGED_MAX_SEQS], resid[KVQ_PAGED_MAX_SEQS], zero[KVQ_PAGED_MAX_SEQS], from[KVQ_PAGED_MAX_SEQS];
  bool any = false;
  for (int b = 0; b < B; ++b) {
    const int L = seq_lens[b];
    if (L < 0 || L > max_seq_len) return KVQ_ERR_ARG;
    if (L > cf.max_tokens) return KVQ_ERR_CAPACITY;
    const int grouped = (R > 0) ? kGroup * ceil_div(std::max(L - R, 0), kGroup) : kGroup * (L / kGroup);
    groups[b] = grouped / kGroup;
    resid[b] = L - grouped;
    from[b] = grouped;
    zero[b] = 0;
    any = any || L > 0;
  }
  if (any && (k == nullptr || v == nullptr)) return KVQ_ERR_NULL;
  if (any && (!aligned(k) || !aligned(v))) return KVQ_ERR_ALIGN;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long src_stride = static_cast<long long>(max_seq_len) * cf.head_dim;
  st = paged_quantize(cache, k, v, src_stride, groups, zero, zero, s);
  if (st != KVQ_OK) return st;
  st = paged_copy(cache, k, v, src_stride, resid, from, zero, s);
  if (st != KVQ_OK) return st;
  for (int b = 0; b < B; ++b) {
    cache->n_grouped[b] = kGroup * groups[b];
    cache->n_resid[b] = resid[b];
  }
  return KVQ_OK;
}

kvq_status kv_paged_append(kivi_paged_cache* cache, const uint16_t* k_new, const uint16_t* v_new, void* stream) {
  kvq_status st = check_paged_cache(cache);
  if (st != KVQ_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_NULL;
  if (!aligned(k_new) || !aligned(v_new)) return KVQ_ERR_ALIGN;
  const kivi_config& cf = cache->pcfg.cfg;
  const int B = cf.batch;
  for (int b = 0; b < B; ++b)
    if (cache->n_grouped[b] + cache->n_resid[b] + 1 > cf.max_tokens) return KVQ_ERR_CAPACITY;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  kivi_paged_cache c = *cache;
  int counts[KVQ_PAGED_MAX_SEQS], one[KVQ_PAGED_MAX_SEQS], zero[KVQ_PAGED_MAX_SEQS], row[KVQ_PAGED_MAX_SEQS];
  bool flush = false;
  for (int b = 0; b < B; ++b) {  // full windows first (R > 0)
    counts[b] = (c.n_resid[b] == c.res_cap) ? c.res_cap / kGroup : 0;
    flush = flush || counts[b] > 0;
  }
  if (flush) {
    st = paged_flush_groups(&c, counts, s);
    if (st != KVQ_OK) return st;
  }
  for (int b = 0; b < B; ++b) {
    one[b] = 1;
    zero[b] = 0;
    row[b] = c.n_resid[b];
  }
  st = paged_copy(&c, k_new, v_new, cf.head_dim, one, zero, row, s);
  if (st != KVQ_OK) return st;
  flush = false;
  for (int b = 0; b < B; ++b) {
    c.n_resid[b] += 1;
    counts[b] = (cf.residual_len == 0 && c.n_resid[b] == kGroup) ? 1 : 0;  // a full 32-slot stage (R = 0)
    flush = flush || counts[b] > 0;
  }
  if (flush) {
    st = paged_flush_groups(&c, counts, s);
    if (st != KVQ_OK) return st;
  }
  *cache = c;
  return KVQ_OK;
}

kvq_status kv_paged_flush(kivi_paged_cache* cache, void* stream) {
  kvq_status st = check_paged_cache(cache);
  if (st != KVQ_OK) return st;
  int counts[KVQ_PAGED_MAX_SEQS];
  bool any = false;
  for (int b = 0; b < cache->pcfg.cfg.batch; ++b) {
    counts[b] = cache->n_resid[b] / kGroup;
    any = any || counts[b] > 0;
  }
  if (!any) return KVQ_OK;
  kivi_paged_cache c = *cache;
  st = paged_flush_groups(&c, counts, static_cast<cudaStream_t>(stream));
  if (st != KVQ_OK) return st;
  *cache = c;
  return KVQ_OK;
}

size_t kv_paged_decode_workspace_bytes(const kivi_paged_config* cfg) {
  if (check_paged_config(cfg) != KVQ_OK) return 0;
  return decode_ws_bytes(cfg->cfg.batch, cfg->cfg.q_heads, cfg->cfg.head_dim);
}

kvq_status kv_paged_decode_attention(const kivi_paged_cache* cache, const uint16_t* q, void* out, int32_t out_fp32,
                                     float softmax_scale, void* ws, size_t ws_bytes, void* stream) {
  kvq_status st = check_paged_cache(cache);
  if (st != KVQ_OK) return st;
  if (q == nullptr || out == nullptr) return KVQ_ERR_NULL;
  if (!aligned(q) || !aligned(out)) return KVQ_ERR_ALIGN;
  if (ws == nullptr) return KVQ_ERR_WORKSPACE;
  if (!aligned(ws)) return KVQ_ERR_ALIGN;
  const kivi_config& cf = cache->pcfg.cfg;
  if (ws_bytes < decode_ws_bytes(cf.batch, cf.q_heads, cf.head_dim)) return KVQ_ERR_WORKSPACE;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return KVQ_ERR_ARG;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cf.head_dim));

  // Units of every (sequence, kv head) pair, one pair after the other, cut
  // into equal stream-K slices: about one slice per resident block, at least
  // kMinUnitsPerSplit units, and at most kMaxSplits - 1 slices over the
  // longest pair (its partials fit the workspace). Each pair is charged
  // kPairLeadUnits more units for the segment a block spends on it (pipeline
  // start, query set-up, partial write and merge), so that blocks whose slice
  // crosses many short sequences get fewer units of work.
  kvq::PagedSeqs seqs{};
  seqs.pools.block_table = cache->block_table;
  seqs.pools.groups_cap = cache->groups_cap;
  seqs.pools.num_blocks = cache->pcfg.num_blocks;
  seqs.n_seqs = cf.batch;
  seqs.pair_lead = kPairLeadUnits;
  long long total = 0;
  int max_u = 0;
  for (int b = 0; b < cf.batch; ++b) {
    const int ng = cache->n_grouped[b] / kGroup, nr = cache->n_resid[b];
    if (ng + nr == 0) return KVQ_ERR_ARG;
    const int U = ng + (use_swapped_decode(cf) ? kvq::kTrChunkUnits : kvq::kChunkUnits) * ceil_div(nr, kGroup);
    seqs.unit0[b] = static_cast<int>(total);
    seqs.n_groups[b] = ng;
    seqs.n_resid[b] = nr;
    total += static_cast<long long>(cf.kv_heads) * (U + kPairLeadUnits);
    if (total > INT_MAX) return KVQ_ERR_UNSUPPORTED;
    max_u = std::max(max_u, U);
  }
  seqs.unit0[cf.batch] = static_cast<int>(total);
  const int per_sm = use_swapped_decode(cf)
                         ? kvq::kivi_paged_decode_tr_blocks_per_sm(cf.head_dim, cf.k_bits, cf.v_bits)
                         : kvq::kivi_paged_decode_blocks_per_sm(cf.head_dim, cf.k_bits, cf.v_bits);
  const long long slots = static_cast<long long>(kvq::device_sm_count()) * std::max(1, per_sm);
  long long per = (total + slots - 1) / slots;
  per = std::max<long long>(per, kMinUnitsPerSplit);
  per = std::max<long long>(per, ceil_div(max_u, kMaxSplits - 1));
  DecodePlan plan{};
  plan.units_per_block = static_cast<int>(per);
  plan.n_blocks = static_cast<int>((total + per - 1) / per);
  plan.part_stride = std::min(kMaxSplits, ceil_div(max_u, per) + 1);

  kivi_cache view{};
  view.cfg = cf;
  view.k_codes = cache->pool;
  view.k_res = cache->k_res;
  view.v_res = cache->v_res;
  view.groups_cap = cache->groups_cap;
  view.res_cap = cache->res_cap;
  const kvq::KiviDecodeArgs a = kivi_decode_args(&view, plan, q, out, out_fp32, scale, static_cast<uint8_t*>(ws));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return from_cuda(use_swapped_decode(cf) ? kvq::launch_kivi_decode_tr_paged(a, seqs, s)
                                          : kvq::launch_kivi_decode_paged(a, seqs, s));
}

size_t fp8_quantize_workspace_bytes(int32_t batch, int32_t kv_heads, int32_t seq_len, int32_t head_dim) {
  (void)batch;
  (void)kv_heads;
  (void)seq_len;
  (void)head_dim;
  return static_cast<size_t>(kAmaxBlocksMax) * sizeof(uint32_t);
}

size_t fp8_pool_bytes(int32_t num_blocks, int32_t kv_heads, int32_t head_dim) {
  if (num_blocks <= 0 || kv_heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
  return static_cast<size_t>(num_blocks) * kv_heads * 16 * head_dim;
}

kvq_status fp8_pool_init(fp8_pool* pool, int32_t role, int32_t fp8_format, int32_t per_head, int32_t num_blocks,
                         int32_t kv_heads, int32_t head_dim, void* buf, float* scale) {
  if (pool == nullptr || buf == nullptr || scale == nullptr) return KVQ_ERR_NULL;
  if (role != KVQ_ROLE_KEY && role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (fp8_format != 0 && fp8_format != 1) return KVQ_ERR_ARG;
  if (per_head != 0 && per_head != 1) return KVQ_ERR_ARG;
  if (num_blocks <= 0 || kv_heads <= 0) return KVQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (!aligned(buf) || !aligned(scale)) return KVQ_ERR_ALIGN;
  fp8_pool p{};
  p.role = role;
  p.fp8_format = fp8_format;
  p.per_head = per_head;
  p.num_blocks = num_blocks;
  p.kv_heads = kv_heads;
  p.head_dim = head_dim;
  p.pool = static_cast<uint8_t*>(buf);
  p.scale = scale;
  *pool = p;
  return KVQ_OK;
}

namespace {
kvq_status check_fp8_pool(const fp8_pool* p) {
  if (p == nullptr || p->pool == nullptr || p->scale == nullptr) return KVQ_ERR_NULL;
  if (p->role != KVQ_ROLE_KEY && p->role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (p->fp8_format != 0 && p->fp8_format != 1) return KVQ_ERR_ARG;
  if (p->per_head != 0 && p->per_head != 1) return KVQ_ERR_ARG;
  if (p->num_blocks <= 0 || p->kv_heads <= 0) return KVQ_ERR_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (!aligned(p->pool) || !aligned(p->scale)) return KVQ_ERR_ALIGN;
  return KVQ_OK;
}
}  // namespace

kvq_status fp8_kv_quantize(const fp8_pool* pool, const uint16_t* x, int32_t batch, int32_t seq_len,
                           const int32_t* block_table, int32_t max_blocks, int32_t static_scale, void* ws,
                           size_t ws_bytes, void* stream) {
  const kvq_status st = check_fp8_pool(pool);
  if (st != KVQ_OK) return st;
  if (x == nullptr || block_table == nullptr) return KVQ_ERR_NULL;
  if (batch <= 0 || seq_len <= 0 || max_blocks <= 0) return KVQ_ERR_ARG;
  if (static_scale != 0 && static_scale != 1) return KVQ_ERR_ARG;
  const int kv_heads = pool->kv_heads, head_dim = pool->head_dim;
  if (pool->per_head && kv_heads > kAmaxBlocksMax) return KVQ_ERR_UNSUPPORTED;
  if (ceil_div(seq_len, 16) > max_blocks) return KVQ_ERR_CAPACITY;
  if (!aligned(x) || !aligned(block_table)) return KVQ_ERR_ALIGN;
  if (!static_scale) {
    if (ws == nullptr) return KVQ_ERR_WORKSPACE;
    if (!aligned(ws)) return KVQ_ERR_ALIGN;
    if (ws_bytes < fp8_quantize_workspace_bytes(batch, kv_heads, seq_len, head_dim)) return KVQ_ERR_WORKSPACE;
  }
  kvq::Fp8QuantArgs a{};
  a.x = x;
  a.batch = batch;
  a.kv_heads = kv_heads;
  a.seq_len = seq_len;
  a.head_dim = head_dim;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.num_blocks = pool->num_blocks;
  a.pool = pool->pool;
  a.scale = pool->scale;
  a.static_scale = static_scale;
  a.per_head = pool->per_head;
  a.fmt = pool->fp8_format;
  // keys in the m16n8k32 order (read by both decode paths), values in p.V's
  a.value_layout = (pool->role == KVQ_ROLE_KEY) ? 2 : 1;
  a.amax_partials = static_cast<uint32_t*>(ws);
  // amax blocks per scale: the partials of all scales fit the workspace, and
  // about 8 blocks per SM run in all
  const int n_scales = pool->per_head ? kv_heads : 1;
  const long long n_vec = static_cast<long long>(batch) * seq_len * head_dim / 8 * (pool->per_head ? 1 : kv_heads);
  a.amax_blocks = static_cast<int>(std::max<long long>(
      1, std::min<long long>({static_cast<long long>(kAmaxBlocksMax / n_scales),
                              (8LL * kvq::device_sm_count() + n_scales - 1) / n_scales, (n_vec + 255) / 256})));
  return from_cuda(kvq::launch_fp8_quantize(a, static_cast<cudaStream_t>(stream)));
}

// FP8 decode workspace: the split-K layout of decode_ws_bytes, then the E4M3
// query (B*Hq*D bytes, rounded to 256), its scale (a 256-byte slot) and the
// amax partials of the query (kQueryAmaxBlocks words).
size_t fp8_query_bytes(int batch, int q_heads, int head_dim) {
  return (static_cast<size_t>(batch) * q_heads * head_dim + 255) / 256 * 256;
}

size_t fp8_decode_ws_bytes(int batch, int q_heads, int head_dim) {
  return decode_ws_bytes(batch, q_heads, head_dim) + fp8_query_bytes(batch, q_heads, head_dim) + 256 +
         static_cast<size_t>(kQueryAmaxBlocks) * sizeof(uint32_t);
}

size_t fp8_decode_workspace_bytes(int32_t batch, int32_t q_heads, int32_t head_dim) {
  if (batch <= 0 || q_heads <= 0 || head_dim <= 0) return 0;
  return fp8_decode_ws_bytes(batch, q_heads, head_dim);
}

kvq_status fp8_decode_attention(const uint16_t* q, const fp8_pool* k, const fp8_pool* v, int32_t q_fp8,
                                const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                                int32_t max_blocks, int32_t max_seq_len, void* out, int32_t out_fp32,
                                float softmax_scale, void* ws, size_t ws_bytes, void* stream) {
  kvq_status st = check_fp8_pool(k);
  if (st != KVQ_OK) return st;
  st = check_fp8_pool(v);
  if (st != KVQ_OK) return st;
  if (k->role != KVQ_ROLE_KEY || v->role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (k->fp8_format != v->fp8_format || k->per_head != v->per_head) return KVQ_ERR_ARG;
  if (k->num_blocks != v->num_blocks || k->kv_heads != v->kv_heads || k->head_dim != v->head_dim) return KVQ_ERR_SHAPE;
  if (!q || !block_table || !seq_lens || !out) return KVQ_ERR_NULL;
  if (batch <= 0 || q_heads <= 0 || max_blocks <= 0 || max_seq_len <= 0) return KVQ_ERR_ARG;
  if (q_fp8 != 0 && q_fp8 != 1) return KVQ_ERR_ARG;
  const int kv_heads = k->kv_heads, head_dim = k->head_dim, block_size = 16;
  if (batch > 65535 || kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  if (q_heads % kv_heads != 0) return KVQ_ERR_SHAPE;
  if (q_heads / kv_heads > kvq::kMaxGqa) return KVQ_ERR_UNSUPPORTED;
  if (max_seq_len > max_blocks * block_size) return KVQ_ERR_CAPACITY;
  if (!aligned(q) || !aligned(block_table) || !aligned(seq_lens) || !aligned(out)) return KVQ_ERR_ALIGN;
  if (ws == nullptr) return KVQ_ERR_WORKSPACE;
  if (!aligned(ws)) return KVQ_ERR_ALIGN;
  if (ws_bytes < fp8_decode_ws_bytes(batch, q_heads, head_dim)) return KVQ_ERR_WORKSPACE;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return KVQ_ERR_ARG;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  const int num_blocks = k->num_blocks, per_head = k->per_head, fp8_format = k->fp8_format;
  const uint8_t* const k_pool = k->pool;
  const uint8_t* const v_pool = v->pool;
  const float* const k_scale = k->scale;
  const float* const v_scale = v->scale;
  const int nblk = ceil_div(max_seq_len, block_size);
  uint8_t* const q_area = static_cast<uint8_t*>(ws) + decode_ws_bytes(batch, q_heads, head_dim);
  uint8_t* const q8 = q_area;
  float* const q_scale = reinterpret_cast<float*>(q_area + fp8_query_bytes(batch, q_heads, head_dim));
  if (q_fp8) {
    kvq::Fp8QueryArgs qa{};
    qa.q = q;
    qa.n = static_cast<long long>(batch) * q_heads * head_dim;
    qa.q8 = q8;
    qa.q_scale = q_scale;
    qa.partials = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(q_scale) + 256);
    qa.amax_blocks = static_cast<int>(std::max<long long>(
        1, std::min<long long>(kQueryAmaxBlocks, (qa.n / 8 + 255) / 256)));
    const kvq_status st = from_cuda(kvq::launch_fp8_quantize_query(qa, static_cast<cudaStream_t>(stream)));
    if (st != KVQ_OK) return st;
  }
  const int splits = choose_splits(nblk, batch * kv_heads, kMaxSplits, kvq::fp8_decode_blocks_per_sm(head_dim), 0);
  kvq::Fp8DecodeArgs a{};
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.per_head = per_head;
  a.fmt = fp8_format;
  a.q_fp8 = q_fp8;
  a.q8 = q8;
  a.q_scale = q_scale;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.q_heads = q_heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.splits = splits;
  a.blocks_per_split = ceil_div(nblk, splits);
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.status = reinterpret_cast<uint32_t*>(base);
  a.counters = reinterpret_cast<uint32_t*>(base + kWsHeader);
  a.part_o = reinterpret_cast<float*>(base + kWsHeader + counters_bytes(batch, q_heads));
  a.part_ml = a.part_o + static_cast<size_t>(batch) * q_heads * splits * head_dim;
  a.out = out;
  a.out_fp32 = out_fp32;
  return from_cuda(kvq::launch_fp8_decode(a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// NVFP4 paged cache
// ---------------------------------------------------------------------------
size_t nvfp4_pool_bytes(int32_t num_blocks, int32_t kv_heads, int32_t head_dim) {
  if (num_blocks <= 0 || kv_heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
  return static_cast<size_t>(num_blocks) * kv_heads * 9 * head_dim;
}

kvq_status nvfp4_pool_init(nvfp4_pool* pool, int32_t role, int32_t num_blocks, int32_t kv_heads, int32_t head_dim,
                           void* buf, float* tensor_scale) {
  if (pool == nullptr || buf == nullptr || tensor_scale == nullptr) return KVQ_ERR_NULL;
  if (role != KVQ_ROLE_KEY && role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (num_blocks <= 0 || kv_heads <= 0) return KVQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (!aligned(buf) || !aligned(tensor_scale)) return KVQ_ERR_ALIGN;
  nvfp4_pool p{};
  p.role = role;
  p.num_blocks = num_blocks;
  p.kv_heads = kv_heads;
  p.head_dim = head_dim;
  p.pool = static_cast<uint8_t*>(buf);
  p.tensor_scale = tensor_scale;
  *pool = p;
  return KVQ_OK;
}

namespace {
kvq_status check_nvfp4_pool(const nvfp4_pool* p) {
  if (p == nullptr || p->pool == nullptr || p->tensor_scale == nullptr) return KVQ_ERR_NULL;
  if (p->role != KVQ_ROLE_KEY && p->role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (p->num_blocks <= 0 || p->kv_heads <= 0) return KVQ_ERR_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (!aligned(p->pool) || !aligned(p->tensor_scale)) return KVQ_ERR_ALIGN;
  return KVQ_OK;
}
}  // namespace

size_t nvfp4_quantize_workspace_bytes(void) { return static_cast<size_t>(kAmaxBlocksMax) * sizeof(uint32_t); }

kvq_status nvfp4_kv_quantize(const nvfp4_pool* pool, const uint16_t* x, int32_t batch, int32_t seq_len,
                             const int32_t* block_table, int32_t max_blocks, int32_t static_scale, void* ws,
                             size_t ws_bytes, void* stream) {
  const kvq_status st = check_nvfp4_pool(pool);
  if (st != KVQ_OK) return st;
  if (x == nullptr || block_table == nullptr) return KVQ_ERR_NULL;
  if (batch <= 0 || seq_len <= 0 || max_blocks <= 0) return KVQ_ERR_ARG;
  if (static_scale != 0 && static_scale != 1) return KVQ_ERR_ARG;
  if (ceil_div(seq_len, 16) > max_blocks) return KVQ_ERR_CAPACITY;
  if (!aligned(x) || !aligned(block_table)) return KVQ_ERR_ALIGN;
  if (!static_scale) {
    if (ws == nullptr) return KVQ_ERR_WORKSPACE;
    if (!aligned(ws)) return KVQ_ERR_ALIGN;
    if (ws_bytes < nvfp4_quantize_workspace_bytes()) return KVQ_ERR_WORKSPACE;
  }
  kvq::Nvfp4QuantArgs a{};
  a.x = x;
  a.batch = batch;
  a.kv_heads = pool->kv_heads;
  a.seq_len = seq_len;
  a.head_dim = pool->head_dim;
  a.role = pool->role;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.num_blocks = pool->num_blocks;
  a.pool = pool->pool;
  a.scale = pool->tensor_scale;
  a.static_scale = static_scale;
  a.amax_partials = static_cast<uint32_t*>(ws);
  const long long n_vec = static_cast<long long>(batch) * pool->kv_heads * seq_len * pool->head_dim / 8;
  a.amax_blocks = static_cast<int>(std::max<long long>(
      1, std::min<long long>({static_cast<long long>(kAmaxBlocksMax), 8LL * kvq::device_sm_count(), (n_vec + 255) / 256})));
  return from_cuda(kvq::launch_nvfp4_quantize(a, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_decode_workspace_bytes(int32_t batch, int32_t q_heads, int32_t head_dim) {
  if (batch <= 0 || q_heads <= 0 || head_dim <= 0) return 0;
  return decode_ws_bytes(batch, q_heads, head_dim);
}

kvq_status nvfp4_decode_attention(const uint16_t* q, const nvfp4_pool* k, const nvfp4_pool* v,
                                  const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                                  int32_t max_blocks, int32_t max_seq_len, void* out, int32_t out_fp32,
                                  float softmax_scale, void* ws, size_t ws_bytes, void* stream) {
  kvq_status st = check_nvfp4_pool(k);
  if (st != KVQ_OK) return st;
  st = check_nvfp4_pool(v);
  if (st != KVQ_OK) return st;
  if (k->role != KVQ_ROLE_KEY || v->role != KVQ_ROLE_VALUE) return KVQ_ERR_ARG;
  if (k->num_blocks != v->num_blocks || k->kv_heads != v->kv_heads || k->head_dim != v->head_dim) return KVQ_ERR_SHAPE;
  if (!q || !block_table || !seq_lens || !out) return KVQ_ERR_NULL;
  if (batch <= 0 || q_heads <= 0 || max_blocks <= 0 || max_seq_len <= 0) return KVQ_ERR_ARG;
  const int kv_heads = k->kv_heads, head_dim = k->head_dim;
  if (batch > 65535 || kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  if (q_heads % kv_heads != 0) return KVQ_ERR_SHAPE;
  if (q_heads / kv_heads > kvq::kMaxGqa) return KVQ_ERR_UNSUPPORTED;
  if (max_seq_len > max_blocks * 16) return KVQ_ERR_CAPACITY;
  if (!aligned(q) || !aligned(block_table) || !aligned(seq_lens) || !aligned(out)) return KVQ_ERR_ALIGN;
  if (ws == nullptr) return KVQ_ERR_WORKSPACE;
  if (!aligned(ws)) return KVQ_ERR_ALIGN;
  if (ws_bytes < decode_ws_bytes(batch, q_heads, head_dim)) return KVQ_ERR_WORKSPACE;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return KVQ_ERR_ARG;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  const int nblk = ceil_div(max_seq_len, 16);
  const int per_sm = kvq::nvfp4_decode_blocks_per_sm(head_dim, q_heads / kv_heads);
  const int splits = choose_splits(nblk, batch * kv_heads, kMaxSplits, per_sm, 0);
  kvq::Nvfp4DecodeArgs a{};
  a.q = q;
  a.k_pool = k->pool;
  a.v_pool = v->pool;
  a.k_scale = k->tensor_scale;
  a.v_scale = v->tensor_scale;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.q_heads = q_heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.max_blocks = max_blocks;
  a.num_blocks = k->num_blocks;
  a.splits = splits;
  a.blocks_per_split = ceil_div(nblk, splits);
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.status = reinterpret_cast<uint32_t*>(base);
  a.counters = reinterpret_cast<uint32_t*>(base + kWsHeader);
  a.part_o = reinterpret_cast<float*>(base + kWsHeader + counters_bytes(batch, q_heads));
  a.part_ml = a.part_o + static_cast<size_t>(batch) * q_heads * splits * head_dim;
  a.out = out;
  a.out_fp32 = out_fp32;
  return from_cuda(kvq::launch_nvfp4_decode(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
// The split-K scratch (status word, split counters, partials) lives in one
// file-scope device array instead of a caller workspace. Every GPU that loads
// this library keeps the array until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// The array's device address on the current device. In host code the array's
// name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached. The first lookup on a device
// also zeroes the array's header (status word and split counters) on
// `stream`, so the status word starts clear; later calls leave it alone.
kvq_status noalloc_scratch_address(void** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kvq_noalloc_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, kWsHeader, stream) != cudaSuccess) return KVQ_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kv_decode_attention_noalloc(const kivi_cache* cache, const uint16_t* q, void* out, int32_t out_fp32,
                                       float softmax_scale, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (q == nullptr || out == nullptr) return KVQ_ERR_NULL;
  if (!aligned(q) || !aligned(out)) return KVQ_ERR_ALIGN;
  if (cache->n_grouped + cache->n_resid == 0) return KVQ_ERR_ARG;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return KVQ_ERR_ARG;
  const kivi_config& cf = cache->cfg;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cf.head_dim));

  const DecodePlan plan = plan_kivi_decode(cache);
  const int splits_total = plan.part_stride;
  const size_t head = static_cast<size_t>(kWsHeader) + counters_bytes(cf.batch, cf.q_heads);
  const size_t need = head + static_cast<size_t>(cf.batch) * cf.q_heads * splits_total *
                                 (static_cast<size_t>(cf.head_dim) + 2) * sizeof(float);
  if (need > static_cast<size_t>(KVQ_NOALLOC_SCRATCH_BYTES)) return KVQ_ERR_CAPACITY;

  void* ws = nullptr;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = noalloc_scratch_address(&ws, s);
  if (st != KVQ_OK) return st;
  // the split counters must start at zero (a call that timed out may have left
  // some set); the status word keeps the error bits of earlier calls
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(base + kWsHeader, 0, head - kWsHeader, s) != cudaSuccess) return KVQ_ERR_CUDA;

  const kvq::KiviDecodeArgs a = kivi_decode_args(cache, plan, q, out, out_fp32, scale, base);
  return from_cuda(launch_contiguous_decode(cf, a, s));
}

kvq_status kv_decode_noalloc_status(uint32_t* status, int32_t clear, void* stream) {
  if (status == nullptr) return KVQ_ERR_NULL;
  void* ws = nullptr;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const kvq_status st = noalloc_scratch_address(&ws, s);
  if (st != KVQ_OK) return st;
  if (cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (clear != 0 && cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return KVQ_ERR_CUDA;
  return (*status & kvq::kStatusTimeout) != 0 ? KVQ_ERR_TIMEOUT : KVQ_OK;
}

}  // extern "C"
