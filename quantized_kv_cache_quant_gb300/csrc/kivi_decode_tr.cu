// KIVI decode attention for caches whose kv heads serve at most four query
// heads (MHA, GQA-2, GQA-4): the roles of the tensor-core operands swapped.
//
// The decode kernel of kivi_kernels.cu puts 8 query heads x {hi, lo} on the 16
// rows of each m16n8k16 tile; with one query head per kv head, 14 of those rows
// are empty. Here the tokens (q . k^T) and the channels (p . V) are the rows
// and the query heads x {hi, lo} the 8 columns, so the same packed codes serve
// as A operands (the extracted registers of one code word are exactly the A
// fragments of two 16-token or two 16-channel tiles) and every group takes 32
// MMAs instead of 64, with half the accumulators. It serves both the contiguous
// cache and the paged one (per-sequence units, groups fetched from the pool
// block of the block table), as the first kernel does.
//
// Method: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 3
// (keys per channel, values per token, groups of 32 tokens, fp16 window);
// attention softmax(q K^T / sqrt(d)) V of "大模型量化从0到1（十三）：KV Cache 量化"
// (CSDN), section 2, with grouped-query sharing (section 5).
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

template <int D, int KB, int VB>
struct KiviTr {
  static constexpr int KS = D / 16;                     // 16-channel k-steps of q . k^T
  static constexpr int MTV = D / 16;                    // 16-channel row tiles of p . V
  static constexpr int NQ = D / 32;                     // value code words per (k-step[, r])
  static constexpr int KW = (KB == 2) ? D / 16 : D / 8;
  static constexpr int VW = (VB == 2) ? D / 16 : D / 8;
  static constexpr int KC = 32 * D * KB / 8;
  static constexpr int KM = 4 * D;
  static constexpr int VC = 32 * D * VB / 8;
  static constexpr int VM = 128;
  static constexpr int STAGE = KC + KM + VC + VM;
};

// Fields of the packed codes read as fp16 subnormals at bits 6-7 / 8-9 (2-bit)
// or 6-9 (4-bit); the multipliers bring code * 2^(P-24) back to code.
constexpr uint32_t kTrMaskP6 = 0x00C000C0u;
constexpr uint32_t kTrMaskP8 = 0x03000300u;
constexpr uint32_t kTrMask4 = 0x03C003C0u;
constexpr float kTrInvP6 = 262144.0f;
constexpr float kTrInvP8 = 65536.0f;

constexpr int kTrStages = 4;

// Sequence state of the contiguous cache (every pair alike); the paged cache
// passes PagedSeqs.
struct TrNoSeqs {};

// Block-table entries a warp of the paged decode keeps in its lanes.
template <bool kPaged>
struct TrTableLanes {
  int tbase = 0, tblk = 0;
};
template <>
struct TrTableLanes<false> {};

// The sequence owning unit x: the b < n with begin[b] <= x < begin[b + 1].
__device__ __forceinline__ int tr_seq_of(const int* begin, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (begin[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

template <int D, int KB, int VB>
struct TrSmem {
  static constexpr int BAR_BYTES = 256;
  static constexpr int STAGE_BYTES = 4 * kTrStages * KiviTr<D, KB, VB>::STAGE;
  static constexpr int O_FLOATS = 4 * 8 * D;
  static constexpr int COMBINE = (O_FLOATS + 64) * 4;
  static constexpr int WIN_ROW = 2 * D + 16;
  static constexpr int AREA = STAGE_BYTES > COMBINE ? STAGE_BYTES : COMBINE;
  static constexpr int BYTES = BAR_BYTES + AREA;
  static_assert(kTrStages * KiviTr<D, KB, VB>::STAGE >= 32 * WIN_ROW, "a warp's stages hold one window chunk");
};

// The online softmax step for query head t = lane % 4 over this thread's four
// scores (tokens g, g + 8, g + 16, g + 24 of the group or chunk), log2 units,
// with the lazy rescale of the decode kernel (the reference maximum moves only
// when a score exceeds it by more than 0.5, so p <= 2^0.5 and p * s fits fp16).
template <int MT>
__device__ __forceinline__ void tr_softmax(const float (&sc)[4], float (&p)[4], float (&o_acc)[MT][4], float& m_run,
                                           float& l_run, float& vz_run) {
  float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  mx = col_max(mx);
  if (mx > m_run + 0.5f) {
    const float alpha = fast_exp2(m_run - mx);
    l_run *= alpha;
    vz_run *= alpha;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      o_acc[i][0] *= alpha;
      o_acc[i][1] *= alpha;
      o_acc[i][2] *= alpha;
      o_acc[i][3] *= alpha;
    }
    m_run = mx;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(sc[i] - m_run);
}

// The fp16 window chunks c_first, c_first + 4, ... < c_end of one warp, with
// the swapped operands: A = the chunk's key rows (ldmatrix) against B = the
// query, then A = the value rows transposed (ldmatrix.trans) against B = p.
// o_acc arrives in code units and leaves in real units. Kept out of line, with
// the accumulators passed by value and returned through o_io. Returns false when
// a copy wait timed out.
template <int D, int VB>
__device__ __noinline__ bool tr_window_chunks(const uint16_t* k_res, const uint16_t* v_res, long long row_base,
                                              int n_resid, int c_first, int c_end, uint8_t* buf, int win_row,
                                              uint64_t* wbar, uint32_t& wphase, const uint32_t (&qb)[D / 16][2],
                                              float p2e_h, float (&o_io)[D / 16][4], float& m_run, float& l_run,
                                              float& vz_run) {
  constexpr int KS = D / 16, MT = D / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2;
  float o_acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    o_acc[mt][0] = o_io[mt][0] * kTrInvP6;
    o_acc[mt][1] = o_io[mt][1] * kTrInvP6;
    o_acc[mt][2] = o_io[mt][2] * (VB == 2 ? kTrInvP8 : kTrInvP6);
    o_acc[mt][3] = o_io[mt][3] * (VB == 2 ? kTrInvP8 : kTrInvP6);
  }
  uint32_t q[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) q[ks][0] = qb[ks][0], q[ks][1] = qb[ks][1];
  bool ok = true;
  for (int c = c_first; c < c_end; c += 4) {
    const int t0 = c * kGroup;
    const int nv = min(kGroup, n_resid - t0);
    const long long row0 = row_base + t0;
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(wbar, nv * D * 2);
    __syncwarp();
    if (lane < nv) bulk_g2s(buf + lane * win_row, k_res + (row0 + lane) * D, D * 2, wbar);
    if (!mbar_wait_bounded(wbar, wphase)) {
      ok = false;
      break;
    }
    wphase ^= 1u;
    // scores: rows = tokens 16 mt + .., columns = query heads (part 0) and zeros (part 1)
    float sacc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t ka[4];
        ldsm_x4(ka, buf + (16 * mt + (lane & 15)) * win_row + (16 * ks + 8 * (lane >> 4)) * 2);
        mma16816(sacc[mt], ka[0], ka[1], ka[2], ka[3], q[ks][0], q[ks][1]);
      }
    }
    // values of the chunk into the same rows; the rows past the window are zeroed
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(wbar, nv * D * 2);
    __syncwarp();
    if (lane < nv) {
      bulk_g2s(buf + lane * win_row, v_res + (row0 + lane) * D, D * 2, wbar);
    } else {
      uint4* zr = reinterpret_cast<uint4*>(buf + lane * win_row);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) zr[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    float sc[4], p[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* s = sacc[k >> 1];
      const float v = (k & 1) ? s[2] + s[3] : s[0] + s[1];
      sc[k] = (g + 8 * k < nv) ? v * p2e_h : -INFINITY;
    }
    tr_softmax<MT>(sc, p, o_acc, m_run, l_run, vz_run);
    uint32_t bt[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half hi = __float2half_rn(p[k]);
      const __half lo = __float2half_rn((p[k] - __half2float(hi)) * kLoGain);
      bt[k] = movm_trans(h2_bits(__halves2half2(hi, lo)));
      l_run += p[k];
    }
    if (!mbar_wait_bounded(wbar, wphase)) {
      ok = false;
      break;
    }
    wphase ^= 1u;
    __syncwarp();  // the zeroed rows of the other lanes
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t va[4];
        ldsm_x4_trans(va, buf + (16 * ks + (lane & 7) + 8 * (lane >> 4)) * win_row +
                              (16 * mt + 8 * ((lane >> 3) & 1)) * 2);
        mma16816(o_acc[mt], va[0], va[1], va[2], va[3], bt[2 * ks], bt[2 * ks + 1]);
      }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o_io[mt][i] = o_acc[mt][i];
  return ok;
}

// 4 resident blocks per SM (113-126 registers). 6 at D = 64 (79 registers) and
// 5 for the paged cache with 2-bit keys at D = 128 (95) also fit without
// spills, but measured slower on GB300: MHA D 64 47.8 -> 52.0 us, paged GQA-4
// 68.5 -> 70.5 us.
template <int D, int KB, int VB, class SeqT>
__global__ void __launch_bounds__(128, 4) kivi_decode_tr_kernel(KiviDecodeArgs a, SeqT seqs) {
  using P = KiviTr<D, KB, VB>;
  constexpr bool kPaged = !std::is_same<SeqT, TrNoSeqs>::value;
  using S = TrSmem<D, KB, VB>;
  constexpr int MT = P::MTV;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* area = smem + S::BAR_BYTES;
  float* o_s = reinterpret_cast<float*>(area);  // [4 warps][8 rows][D]
  float* m_s = o_s + S::O_FLOATS;               // [4][8]
  float* l_s = m_s + 32;                        // [4][8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int gq = a.q_heads / a.kv_heads;
  // column roles (B operands): column g is query head g / 2, part g % 2 (0: hi, 1: lo);
  // row roles (scores, outputs): this thread's query head is tig
  const int jq = g >> 1, part = g & 1;
  constexpr int GPS = 2, NS = kTrStages / GPS;
  constexpr int SLOT = GPS * P::STAGE;
  uint64_t* bar = bars + warp * kTrStages;
  uint64_t* wbar = bars + 4 * kTrStages + warp;
  uint8_t* ring = area + warp * kTrStages * P::STAGE;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
    mbar_init(wbar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  long long all_units = static_cast<long long>(a.n_pairs) * a.pair_stride;
  if constexpr (kPaged) all_units = seqs.unit0[seqs.n_seqs];
  const long long u0 = static_cast<long long>(blockIdx.x) * a.units_per_block;
  const long long u1 = min(all_units, u0 + a.units_per_block);
  int jg = 0;
  uint32_t wphase = 0;
  bool timed_out = false;
  for (long long u = u0; u < u1;) {
    int pair, upp, n_grp, n_res;
    long long pbase;
    if constexpr (kPaged) {
      // pair (b, h) spans pair_lead units of no work, then its groups and chunks
      const int sb = tr_seq_of(seqs.unit0, seqs.n_seqs, u);
      n_grp = seqs.n_groups[sb];
      n_res = seqs.n_resid[sb];
      upp = n_grp + kTrChunkUnits * ((n_res + kGroup - 1) / kGroup);
      const int span = upp + seqs.pair_lead;
      const int hh = static_cast<int>((u - seqs.unit0[sb]) / span);
      pair = sb * a.kv_heads + hh;
      const long long vbase = seqs.unit0[sb] + static_cast<long long>(hh) * span;
      pbase = vbase + seqs.pair_lead;
      u = vbase + span;
    } else {
      pair = static_cast<int>(u / a.pair_stride);
      pbase = static_cast<long long>(pair) * a.pair_stride;
      upp = a.units_per_pair;
      n_grp = a.n_groups;
      n_res = a.n_resid;
      u = pbase + a.pair_stride;
    }
    const int lo = static_cast<int>(u0 > pbase ? u0 - pbase : 0LL);
    const int hi = static_cast<int>(min(static_cast<long long>(upp), u1 - pbase));
    if (lo >= upp) continue;  // padding after the pair's units (the same for the whole block)
    if constexpr (kPaged) {
      if (hi <= 0) continue;  // the slice ends inside the pair's lead-in: no work here
    }
    const int b = pair / a.kv_heads, h = pair % a.kv_heads;
    const long long bh = pair;
    const int first_block = static_cast<int>(pbase / a.units_per_block);
    const int split = static_cast<int>(blockIdx.x) - first_block;
    const int n_splits = static_cast<int>((pbase + upp - 1) / a.units_per_block) - first_block + 1;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    const int n_chunks = (n_res + kGroup - 1) / kGroup;
    const int g_begin = min(n_grp, lo);
    const int g_end = min(n_grp, hi);
    const int c_begin = min(n_chunks, max(0, lo - n_grp + kTrChunkUnits - 1) / kTrChunkUnits);
    const int c_end = min(n_chunks, max(0, hi - n_grp + kTrChunkUnits - 1) / kTrChunkUnits);

    float m_run = -INFINITY, l_run = 0.0f, vz_run = 0.0f;
    float o_acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;

    const int n_here = g_end - g_begin;
    int n_mine = 0;
    if (!timed_out && n_here > GPS * warp) {
      const int np = (n_here - GPS * warp + 4 * GPS - 1) / (4 * GPS);
      n_mine = GPS * (np - 1) + min(GPS, n_here - GPS * (warp + 4 * (np - 1)));
    }
    const int n_slots = (n_mine + GPS - 1) / GPS;
    // contiguous: the pair's records, groups one after the other
    const long long rec0 = bh * a.groups_cap;
    const uint8_t* kc_g = a.k_codes + rec0 * P::KC;
    const uint8_t* km_g = a.k_meta + rec0 * P::KM;
    const uint8_t* vc_g = a.v_codes + rec0 * P::VC;
    const uint8_t* vm_g = a.v_meta + rec0 * P::VM;
    // paged: group j's pool blocks from the block table through the lanes (lane l
    // holds the entry of the warp's group tbase + l, clamped into the pool)
    TrTableLanes<kPaged> tl;
    auto load_table = [&](int base) {  // warp-wide
      if constexpr (kPaged) {
        tl.tbase = base;
        const int jl = base + lane;
        if (jl < n_mine) {
          const int grp = g_begin + GPS * (warp + 4 * (jl / GPS)) + jl % GPS;
          tl.tblk = min(max(__ldg(seqs.pools.block_table + static_cast<long long>(b) * a.groups_cap + grp), 0),
                        seqs.pools.num_blocks - 1);
        }
      }
    };
    auto slot_blocks = [&](int k, int& b0, int& b1) {  // warp-wide
      if constexpr (kPaged) {
        if (GPS * k + GPS > tl.tbase + 32) load_table(GPS * k);
        b0 = __shfl_sync(0xffffffffu, tl.tblk, GPS * k - tl.tbase);
        b1 = __shfl_sync(0xffffffffu, tl.tblk, GPS * k + 1 - tl.tbase);
      }
    };
    // slot k (groups g_begin + GPS * (warp + 4k) + {0, 1}) through ring position (jg + k) % NS
    auto issue = [&](int k, int b0 = 0, int b1 = 0) {
      const int grp = g_begin + GPS * (warp + 4 * k);
      const uint32_t cnt = static_cast<uint32_t>(min(GPS, g_end - grp));
      uint8_t* dst = ring + ((jg + k) % NS) * SLOT;
      uint64_t* bb = &bar[(jg + k) % NS];
      mbar_arrive_expect_tx(bb, cnt * P::STAGE);
      if constexpr (kPaged) {
        // one copy per group: kv head h's entry of its pool block (the pool is a.k_codes)
        static_assert(GPS == 2, "two blocks per slot");
        const uint8_t* pool_h = a.k_codes + static_cast<long long>(h) * P::STAGE;
        bulk_g2s(dst, pool_h + static_cast<long long>(b0) * a.kv_heads * P::STAGE, P::STAGE, bb);
        if (cnt > 1) bulk_g2s(dst + P::STAGE, pool_h + static_cast<long long>(b1) * a.kv_heads * P::STAGE, P::STAGE, bb);
      } else {
        bulk_g2s(dst, kc_g + grp * static_cast<long long>(P::KC), cnt * P::KC, bb);
        bulk_g2s(dst + GPS * P::KC, km_g + grp * static_cast<long long>(P::KM), cnt * P::KM, bb);
        bulk_g2s(dst + GPS * (P::KC + P::KM), vc_g + grp * static_cast<long long>(P::VC), cnt * P::VC, bb);
        bulk_g2s(dst + GPS * (P::KC + P::KM + P::VC), vm_g + grp * static_cast<long long>(P::VM), cnt * P::VM, bb);
      }
    };
    auto wait_slot = [&](int k) { return mbar_wait_bounded(&bar[(jg + k) % NS], ((jg + k) / NS) & 1); };
    // the records of group j of the warp (paged: each group's four records back
    // to back; contiguous: the GPS groups' records of one kind together)
    auto slot_base = [&](int j) { return ring + ((jg + j / GPS) % NS) * SLOT; };
    auto kc_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE;
      else return slot_base(j) + (j % GPS) * P::KC;
    };
    auto km_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC;
      else return slot_base(j) + GPS * P::KC + (j % GPS) * P::KM;
    };
    auto vc_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC + P::KM;
      else return slot_base(j) + GPS * (P::KC + P::KM) + (j % GPS) * P::VC;
    };
    auto vm_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC + P::KM + P::VC;
      else return slot_base(j) + GPS * (P::KC + P::KM + P::VC) + (j % GPS) * P::VM;
    };
    if constexpr (kPaged) {
      if (n_mine > 0) load_table(0);
      for (int k = 0; k < NS && k < n_slots; ++k) {
        int b0 = 0, b1 = 0;
        slot_blocks(k, b0, b1);
        if (lane == 0) issue(k, b0, b1);
      }
    } else {
      if (lane == 0) {
        for (int k = 0; k < NS && k < n_slots; ++k) issue(k);
      }
    }

    // The query of column g (head jq), channels 16ks + 2tig, +1 and 16ks + 8 + 2tig, +1,
    // scaled by 2^-e (e from the head's largest |q|) so that q * s stays in the fp16 range.
    const bool col_ok = jq < gq;
    const __half* qrow = reinterpret_cast<const __half*>(a.q) +
                         (static_cast<long long>(b) * a.q_heads + h * gq + (col_ok ? jq : 0)) * D;
    float2 qv[P::KS][2];
    float qmax = 0.0f;
#pragma unroll
    for (int ks = 0; ks < P::KS; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __half2 v = col_ok ? *reinterpret_cast<const __half2*>(qrow + 16 * ks + 8 * j + 2 * tig)
                                 : __float2half2_rn(0.0f);
        qv[ks][j] = __half22float2(v);
        qmax = fmaxf(qmax, fmaxf(fabsf(qv[ks][j].x), fabsf(qv[ks][j].y)));
      }
    qmax = quad_max(qmax);
    int e = 0;
    if (qmax > 0.0f) frexpf(qmax, &e);
    const float qscale = ldexpf(1.0f, -e);
    uint32_t qs[P::KS][2];
#pragma unroll
    for (int ks = 0; ks < P::KS; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j) qs[ks][j] = pack_rn_f16x2(qv[ks][j].x * qscale, qv[ks][j].y * qscale);
    const float p2e_q = ldexpf(1.0f, e) * a.scale_log2;
    // the same factor for this thread's row head tig (column 2 tig is lane 8 tig's head)
    const float p2e_h = __shfl_sync(0xffffffffu, p2e_q, 8 * tig);
    const float mult6 = kTrInvP6 * p2e_h, mult8 = (KB == 2 ? kTrInvP8 : kTrInvP6) * p2e_h;

    // q . k_hat of group jj: the thread's scores of head tig, tokens g, g + 8, g + 16, g + 24
    auto qk_scores = [&](int jj, float (&sc)[4]) {
      const uint4* kcw = reinterpret_cast<const uint4*>(kc_of(jj));
      const uint4* kmr = reinterpret_cast<const uint4*>(km_of(jj));
      uint32_t kw[P::KW];
#pragma unroll
      for (int c = 0; c < P::KW / 4; ++c) {
        const uint4 x = kcw[c * 32 + lane];
        kw[4 * c] = x.x;
        kw[4 * c + 1] = x.y;
        kw[4 * c + 2] = x.z;
        kw[4 * c + 3] = x.w;
      }
      float sacc[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
      float bsum = 0.0f;
#pragma unroll
      for (int ks = 0; ks < P::KS; ++ks) {
        const uint4 md = kmr[ks * 4 + tig];  // {s(d0,d0+1), s(d0+8,d0+9), z(d0,d0+1), z(d0+8,d0+9)}
        const __half2 q0 = bits_h2(qs[ks][0]), q1 = bits_h2(qs[ks][1]);
        const __half2 hi0 = __hmul2(q0, bits_h2(md.x));
        const __half2 hi1 = __hmul2(q1, bits_h2(md.y));
        const uint32_t b0 = part ? h2_bits(__hfma2(q0, bits_h2(md.x), __hneg2(hi0))) : h2_bits(hi0);
        const uint32_t b1 = part ? h2_bits(__hfma2(q1, bits_h2(md.y), __hneg2(hi1))) : h2_bits(hi1);
        bsum = dot2_f16_f32(qs[ks][0], md.z, dot2_f16_f32(qs[ks][1], md.w, bsum));
        if constexpr (KB == 2) {
          const uint32_t w = kw[ks];
          const uint32_t l4 = w << 4, r4 = w >> 4, sw = __byte_perm(w, 0u, 0x2301u);
          mma16816(sacc[0], l4 & kTrMaskP6, l4 & kTrMaskP8, r4 & kTrMaskP6, r4 & kTrMaskP8, b0, b1);
          mma16816(sacc[1], w & kTrMaskP6, w & kTrMaskP8, sw & kTrMaskP6, sw & kTrMaskP8, b0, b1);
        } else {
          const uint32_t w0 = kw[2 * ks], w1 = kw[2 * ks + 1];
          mma16816(sacc[0], (w0 << 6) & kTrMask4, (w0 << 2) & kTrMask4, (w1 << 6) & kTrMask4, (w1 << 2) & kTrMask4,
                   b0, b1);
          mma16816(sacc[1], (w0 >> 2) & kTrMask4, (w0 >> 6) & kTrMask4, (w1 >> 2) & kTrMask4, (w1 >> 6) & kTrMask4,
                   b0, b1);
        }
      }
      // q . z of head jq (quad sum over the channels), moved to the lanes whose row head it is
      const float bias = __shfl_sync(0xffffffffu, quad_sum(bsum) * p2e_q, 8 * tig);
      sc[0] = fmaf(sacc[0][0] + sacc[0][1], mult6, bias);
      sc[1] = fmaf(sacc[0][2] + sacc[0][3], mult8, bias);
      sc[2] = fmaf(sacc[1][0] + sacc[1][1], mult6, bias);
      sc[3] = fmaf(sacc[1][2] + sacc[1][3], mult8, bias);
    };

    // One group at a time: q . k^T, softmax and p . V of group j (issuing
    // q . k^T of group j + 1 inside group j's p . V, as the other kernel does,
    // measured 2-3 % slower here: MHA 4K 41.6 against 43.0 us).
    int j = 0;
    float sc[4];
    for (; !timed_out && j < n_mine; ++j) {
      if (j % GPS == 0 && !wait_slot(j / GPS)) {
        timed_out = true;
        break;
      }
      qk_scores(j, sc);
      const uint4* vcw = reinterpret_cast<const uint4*>(vc_of(j));
      const uint4* vmr = reinterpret_cast<const uint4*>(vm_of(j));

      float p[4];
      tr_softmax<MT>(sc, p, o_acc, m_run, l_run, vz_run);

      // p' = p * s_t split into fp16 hi + lo * kLoGain (columns 2 tig, 2 tig + 1 of the
      // token row), transposed into the B fragments of p . V; the scales and
      // zero points of tokens g + 8k are halves 2k + (g & 1) of records g / 2 and 4 + g / 2
      const uint4 vs = vmr[g >> 1], vz = vmr[4 + (g >> 1)];
      const uint32_t vsw[4] = {vs.x, vs.y, vs.z, vs.w};
      const uint32_t vzw[4] = {vz.x, vz.y, vz.z, vz.w};
      uint32_t bt[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 sf = __half22float2(bits_h2(vsw[k]));
        const float2 zf = __half22float2(bits_h2(vzw[k]));
        const float s_t = (g & 1) ? sf.y : sf.x, z_t = (g & 1) ? zf.y : zf.x;
        const float pp = p[k] * s_t;
        const __half hi = __float2half_rn(pp);
        const __half lo = __float2half_rn((pp - __half2float(hi)) * kLoGain);
        bt[k] = movm_trans(h2_bits(__halves2half2(hi, lo)));
        l_run += p[k];
        vz_run = fmaf(p[k], z_t, vz_run);
      }


      // ---- o^T += codes^T . p' (group j): rows = channels 16 mt + .., columns = heads x {hi, lo} ----
      uint32_t vw[P::VW];
#pragma unroll
      for (int c = 0; c < P::VW / 4; ++c) {
        const uint4 x = vcw[c * 32 + lane];
        vw[4 * c] = x.x;
        vw[4 * c + 1] = x.y;
        vw[4 * c + 2] = x.z;
        vw[4 * c + 3] = x.w;
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t B0 = bt[2 * ks], B1 = bt[2 * ks + 1];
#pragma unroll
        for (int q = 0; q < P::NQ; ++q) {
          if constexpr (VB == 2) {
            const uint32_t w = vw[ks * P::NQ + q];
            const uint32_t l4 = w << 4, r4 = w >> 4, sw = __byte_perm(w, 0u, 0x2301u);
            mma16816(o_acc[2 * q], l4 & kTrMaskP6, l4 & kTrMaskP8, r4 & kTrMaskP6, r4 & kTrMaskP8, B0, B1);
            mma16816(o_acc[2 * q + 1], w & kTrMaskP6, w & kTrMaskP8, sw & kTrMaskP6, sw & kTrMaskP8, B0, B1);
          } else {
            const uint32_t w0 = vw[(2 * ks) * P::NQ + q], w1 = vw[(2 * ks + 1) * P::NQ + q];
            mma16816(o_acc[2 * q], (w0 << 6) & kTrMask4, (w0 << 2) & kTrMask4, (w1 << 6) & kTrMask4,
                     (w1 << 2) & kTrMask4, B0, B1);
            mma16816(o_acc[2 * q + 1], (w0 >> 2) & kTrMask4, (w0 >> 6) & kTrMask4, (w1 >> 2) & kTrMask4,
                     (w1 >> 6) & kTrMask4, B0, B1);
          }
        }
      }

      if (j % GPS == GPS - 1 || j + 1 == n_mine) {
        __syncwarp();
        if constexpr (kPaged) {
          const int kn = j / GPS + NS;
          if (kn < n_slots) {
            int b0 = 0, b1 = 0;
            slot_blocks(kn, b0, b1);
            if (lane == 0) {
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              issue(kn, b0, b1);
            }
          }
        } else {
          if (lane == 0 && j / GPS + NS < n_slots) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(j / GPS + NS);
          }
        }
      }
    }

    // ------------------------ fp16 window, 32-token chunks ------------------------
    bool real_units = false, win_pending = false, seg_timeout = timed_out && n_mine > 0;
    if (!timed_out && c_begin + warp < c_end) {
      real_units = true;
      float o_io[MT][4], st[3] = {m_run, l_run, vz_run};
      uint32_t qb[P::KS][2];
#pragma unroll
      for (int i = 0; i < MT; ++i)
        o_io[i][0] = o_acc[i][0], o_io[i][1] = o_acc[i][1], o_io[i][2] = o_acc[i][2], o_io[i][3] = o_acc[i][3];
      // B of q . k^T over fp16 keys: the query itself in the part-0 columns, zero in the part-1 columns
#pragma unroll
      for (int ks = 0; ks < P::KS; ++ks) qb[ks][0] = part ? 0u : qs[ks][0], qb[ks][1] = part ? 0u : qs[ks][1];
      uint32_t ph = wphase;
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the window is complete (see the launch)
      const bool ok = tr_window_chunks<D, VB>(a.k_res, a.v_res, bh * a.res_cap, n_res, c_begin + warp, c_end, ring,
                                              S::WIN_ROW, wbar, ph, qb, p2e_h, o_io, st[0], st[1], st[2]);
#pragma unroll
      for (int i = 0; i < MT; ++i)
        o_acc[i][0] = o_io[i][0], o_acc[i][1] = o_io[i][1], o_acc[i][2] = o_io[i][2], o_acc[i][3] = o_io[i][3];
      m_run = st[0];
      l_run = st[1];
      vz_run = st[2];
      wphase = ph;
      if (!ok) {
        timed_out = true;
        seg_timeout = true;
        win_pending = true;
      }
    }

    if (seg_timeout) {
      if (lane == 0) report_timeout(a.status);
      for (int k = j / GPS; k < n_slots && k < j / GPS + NS; ++k) (void)wait_slot(k);
      if (win_pending) (void)mbar_wait_bounded(wbar, wphase);
    }
    if (timed_out) {
      m_run = -INFINITY;
      l_run = 0.0f;
      vz_run = 0.0f;
#pragma unroll
      for (int i = 0; i < MT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
    }
    jg += n_slots;
    l_run = col_sum(l_run);
    vz_run = col_sum(vz_run);
    __syncthreads();  // every warp is done with its stages; the area is reused below
    // row head tig: channel 16 mt + g (column pair c0 + c1) and 16 mt + 8 + g (c2 + c3)
    const float om_lo = real_units ? 1.0f : kTrInvP6;
    const float om_hi = real_units ? 1.0f : (VB == 2 ? kTrInvP8 : kTrInvP6);
    float* orow = o_s + (warp * 8 + tig) * D;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      orow[16 * mt + g] = fmaf(fmaf(o_acc[mt][1], kLoGainInv, o_acc[mt][0]), om_lo, vz_run);
      orow[16 * mt + 8 + g] = fmaf(fmaf(o_acc[mt][3], kLoGainInv, o_acc[mt][2]), om_hi, vz_run);
    }
    if (g == 0) {
      m_s[warp * 8 + tig] = m_run;
      l_s[warp * 8 + tig] = l_run;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    finish_split<D>(o_s, m_s, l_s, gq, static_cast<long long>(b) * a.q_heads + h * gq, split, n_splits,
                    a.part_stride, a.part_o, a.part_ml, a.counters + bh, a.out, a.out_fp32);
  }
}

template <int D, int KB, int VB, class SeqT>
int tr_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    constexpr int smem = TrSmem<D, KB, VB>::BYTES;
    auto kern = kivi_decode_tr_kernel<D, KB, VB, SeqT>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, smem) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launched as a programmatic dependent of the kernel before it, as the decode
// of kivi_kernels.cu is: the grouped loop reads only group records and q, the
// fp16 window and the workspace are touched after griddepcontrol.wait.
template <int D, int KB, int VB, class SeqT>
cudaError_t tr_dispatch(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  constexpr int smem = TrSmem<D, KB, VB>::BYTES;
  auto kern = kivi_decode_tr_kernel<D, KB, VB, SeqT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_blocks));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, seqs);
}

template <class SeqT>
cudaError_t tr_by_key(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  switch (a.head_dim * 100 + a.k_bits * 10 + a.v_bits) {
    case 6422: return tr_dispatch<64, 2, 2>(a, seqs, s);
    case 6424: return tr_dispatch<64, 2, 4>(a, seqs, s);
    case 6442: return tr_dispatch<64, 4, 2>(a, seqs, s);
    case 6444: return tr_dispatch<64, 4, 4>(a, seqs, s);
    case 12822: return tr_dispatch<128, 2, 2>(a, seqs, s);
    case 12824: return tr_dispatch<128, 2, 4>(a, seqs, s);
    case 12842: return tr_dispatch<128, 4, 2>(a, seqs, s);
    case 12844: return tr_dispatch<128, 4, 4>(a, seqs, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class SeqT>
int tr_occupancy_by_key(int head_dim, int k_bits, int v_bits) {
  switch (head_dim * 100 + k_bits * 10 + v_bits) {
    case 6422: return tr_occupancy<64, 2, 2, SeqT>();
    case 6424: return tr_occupancy<64, 2, 4, SeqT>();
    case 6442: return tr_occupancy<64, 4, 2, SeqT>();
    case 6444: return tr_occupancy<64, 4, 4, SeqT>();
    case 12822: return tr_occupancy<128, 2, 2, SeqT>();
    case 12824: return tr_occupancy<128, 2, 4, SeqT>();
    case 12842: return tr_occupancy<128, 4, 2, SeqT>();
    case 12844: return tr_occupancy<128, 4, 4, SeqT>();
    default: return 1;
  }
}

}  // namespace

cudaError_t launch_kivi_decode_tr(const KiviDecodeArgs& a, cudaStream_t s) { return tr_by_key(a, TrNoSeqs{}, s); }

cudaError_t launch_kivi_decode_tr_paged(const KiviDecodeArgs& a, const PagedSeqs& seqs, cudaStream_t s) {
  return tr_by_key(a, seqs, s);
}

int kivi_decode_tr_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return tr_occupancy_by_key<TrNoSeqs>(head_dim, k_bits, v_bits);
}

int kivi_paged_decode_tr_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return tr_occupancy_by_key<PagedSeqs>(head_dim, k_bits, v_bits);
}

}  // namespace kvq
