// Split-K decode attention over the packed KIVI cache for sm_103a: q . k^T on
// the warp-level tensor-core MMA (mma.sync m16n8k16, the per-group scaled
// query in registers), p . V on the fifth-generation tensor cores (tcgen05.mma
// with the value codes and the accumulators in tensor memory), and the
// log-sum-exp merge of the split partials.
//
// Method: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 3
// (keys per channel, values per token, groups of 32 tokens, fp16 residual
// window); affine dequantization of "大模型量化从0到1（十三）：KV Cache 量化"
// (CSDN), section 10; attention softmax(q K^T / sqrt(d)) V of the same page,
// section 2, with grouped-query sharing (section 5).
//
// Dequantization folded into the contractions (algebra, exact in real numbers):
//   q . k_hat_t = sum_d (q_d s_{g,d}) c_{t,d} + sum_d q_d z_{g,d}
//   sum_t p_t v_hat_{t,d} = sum_t (p_t s_t) c_{t,d} + sum_t p_t z_t
// so the 2/4-bit codes enter the tensor cores as exact fp16 operands.
#include <cmath>
#include <type_traits>

#include "kivi_layout.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Tensor memory of one thread block (128 lanes = the channels of p . V):
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColA = 0;    // 4 group slots x 16 columns: value codes, A of p . V
constexpr uint32_t kColD6 = 64;  // accumulators of codes read at bits 6-7 / 6-9 (units 2^-18)
constexpr uint32_t kColD8 = 80;  // accumulators of 2-bit codes read at bits 8-9 (units 2^-16)
constexpr uint32_t kColDW = 96;  // accumulators of the fp16 window (real units)
constexpr int kTmemBlocksPerSm = 512 / kTmemCols;

// B operand of p . V for one group: 16 rows (8 query heads x {hi, lo} fp16
// parts of p * s_t) x 32 tokens, K-major core matrices of 8 rows x 8 tokens:
// core (n_blk, k_blk) at n_blk * kSbo + k_blk * kLbo. k-step s (tokens 16s ..
// 16s + 15) starts at byte 256 s.
constexpr uint32_t kLbo = 128, kSbo = 512;
constexpr int kBSlot = 1024;

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int KB, int VB>
struct TcSmem {
  using P = Kivi<D, KB, VB>;
  static constexpr int ROUND = 4 * P::STAGE;  // the records of one round (4 groups)
  static constexpr int NS = (49152 / ROUND) < 2 ? 2 : ((49152 / ROUND) > 4 ? 4 : 49152 / ROUND);
  static constexpr int WIN_ROW = 2 * D + 16;  // one fp16 window row, padded: ldmatrix rows hit distinct banks
  static constexpr int WIN_BYTES = 2 * 32 * WIN_ROW;
  static constexpr int OUT_BYTES = (8 * D + 8 * kMaxSplits + 8) * 4;
  static constexpr int AREA = cmax(NS * ROUND, cmax(WIN_BYTES, OUT_BYTES));
  static constexpr int B_BYTES = 2 * 4 * kBSlot;  // two buffers: a batch writes one while the last one's MMAs read the other
  static constexpr int BYTES = B_BYTES + AREA;
};

// Sequence state of the contiguous cache: every pair has a.n_groups groups and
// a.n_resid window tokens, at unit p * pair_stride.
struct NoSeqs {};

// Block-table entries warp 1 keeps in its lanes for the paged decode (nothing
// for the contiguous cache).
template <bool kPaged>
struct TableLanes {
  int tbase = -1024, tblk = 0;
};
template <>
struct TableLanes<false> {};

// Value codes of one group, channel ch (this lane), into 16 tensor-memory
// columns: column j = tokens 2j (low half) and 2j + 1, the code field at bits
// 6-7 (columns 0-7 of 2-bit codes, and every 4-bit column) or 8-9 (columns
// 8-15 of 2-bit codes) of each fp16 half.
// vc: shared address of this channel's VB words.
template <int VB>
__device__ __forceinline__ void fill_value_codes(uint32_t vc, uint32_t taddr) {
  if constexpr (VB == 2) {
    const uint2 x = lds64(vc);
    const uint32_t a = x.x, al = a << 4, ar = a >> 4, as = __byte_perm(a, 0u, 0x2301u);
    const uint32_t b = x.y, bl = b << 4, br = b >> 4, bs = __byte_perm(b, 0u, 0x2301u);
    tmem_st8(taddr, a & kMaskP6, al & kMaskP6, ar & kMaskP6, as & kMaskP6, b & kMaskP6, bl & kMaskP6, br & kMaskP6,
             bs & kMaskP6);
    tmem_st8(taddr + 8, a & kMaskP8, al & kMaskP8, ar & kMaskP8, as & kMaskP8, b & kMaskP8, bl & kMaskP8,
             br & kMaskP8, bs & kMaskP8);
  } else {
    const uint4 x = lds128(vc);
    tmem_st8(taddr, (x.x << 6) & kMask4, (x.x << 2) & kMask4, (x.x >> 2) & kMask4, (x.x >> 6) & kMask4,
             (x.y << 6) & kMask4, (x.y << 2) & kMask4, (x.y >> 2) & kMask4, (x.y >> 6) & kMask4);
    tmem_st8(taddr + 8, (x.z << 6) & kMask4, (x.z << 2) & kMask4, (x.z >> 2) & kMask4, (x.z >> 6) & kMask4,
             (x.w << 6) & kMask4, (x.w << 2) & kMask4, (x.w >> 2) & kMask4, (x.w >> 6) & kMask4);
  }
}

// fp16 window values of channel ch for the 32 tokens of one chunk (rows of
// row_bytes bytes; rows at or past nv read as zero) into 16 columns.
__device__ __forceinline__ void fill_window_values(const uint8_t* rows, int row_bytes, int nv, int ch, uint32_t taddr) {
  const uint16_t* col = reinterpret_cast<const uint16_t*>(rows) + ch;
  const int stride = row_bytes / 2;
  uint32_t r[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t a0 = (2 * j < nv) ? col[(2 * j) * stride] : 0u;
    const uint32_t a1 = (2 * j + 1 < nv) ? col[(2 * j + 1) * stride] : 0u;
    r[j] = a0 | (a1 << 16);
  }
  tmem_st16(taddr, r);
}

// Softmax weights of one group against the reference m_ref (log2 units) and
// the B operand of p . V: this thread's 8 scores sc (query head g, tokens
// 8nt + 2tig + {0, 1}) give p = 2^(sc - m_ref); p * s_t split exactly into
// fp16 hi (row g) + lo (row 8 + g) is stored at k-block nt. Adds sum p and
// sum p z_t to lsum and vzsum.
__device__ __forceinline__ void group_weights(const float (&sc)[8], float m_ref, uint32_t vm, uint32_t brow, int tig,
                                              float& lsum, float& vzsum) {
  // vm: shared address of the group's value meta; brow: this thread's row
  // word in k-block 0 of the B slot (g * 16 + tig * 4 from the slot start)
  const uint4 vs = lds128(vm + tig * 16), vz = lds128(vm + 64 + tig * 16);
  const uint32_t vsw[4] = {vs.x, vs.y, vs.z, vs.w};
  const uint32_t vzw[4] = {vz.x, vz.y, vz.z, vz.w};
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const float p0 = fast_exp2(sc[2 * nt] - m_ref), p1 = fast_exp2(sc[2 * nt + 1] - m_ref);
    const float2 sf = __half22float2(bits_h2(vsw[nt]));
    const float2 zf = __half22float2(bits_h2(vzw[nt]));
    const float pp0 = p0 * sf.x, pp1 = p1 * sf.y;
    const __half2 hh = __floats2half2_rn(pp0, pp1);
    const float2 hf = __half22float2(hh);
    sts32(brow + nt * kLbo, h2_bits(hh));
    sts32(brow + nt * kLbo + kSbo, pack_rn_f16x2(pp0 - hf.x, pp1 - hf.y));
    lsum += p0 + p1;
    vzsum = fmaf(p0, zf.x, fmaf(p1, zf.y, vzsum));
  }
}

// The same for this warp's 8 tokens of a window chunk (k-block kb): 2 scores
// per thread, p split into fp16 hi + lo (the window values are fp16 as stored).
__device__ __forceinline__ void window_weights(const float (&sc)[2], float m_ref, uint8_t* bslot, int kb, int g,
                                               int tig, float& lsum) {
  const float p0 = fast_exp2(sc[0] - m_ref), p1 = fast_exp2(sc[1] - m_ref);
  const __half2 hh = __floats2half2_rn(p0, p1);
  const float2 hf = __half22float2(hh);
  uint8_t* row = bslot + kb * kLbo + g * 16 + tig * 4;
  *reinterpret_cast<uint32_t*>(row) = h2_bits(hh);
  *reinterpret_cast<uint32_t*>(row + kSbo) = pack_rn_f16x2(p0 - hf.x, p1 - hf.y);
  lsum += p0 + p1;
}

// Grid: a 1-D list of 128-thread blocks, at most as many as the GPU keeps
// resident, each with the slice [blockIdx.x * U, (blockIdx.x + 1) * U) of the
// work units of all (batch row, kv head) pairs (units: a pair's groups, then
// its fp16 window cut into 32-token chunks of kChunkUnits units). A block
// takes its groups in rounds of four, group i of a round to warp i:
//   1. the round's records arrive in one shared-memory stage (bulk copies,
//      one mbarrier per stage, a ring of NS stages filled NS rounds ahead);
//   2. warp i: q . k^T of its group on mma.sync (M = 8 query heads x {hi, lo}
//      parts of q * s_{g,d}, N = tokens, B = the key codes as fp16
//      subnormals), q . z on the FMA pipe;
//   3. every warp: the value codes of its 32 channels of all four groups into
//      tensor memory (A of p . V: lane = channel, column = token pair);
//   4. warp i: softmax weights against the block's reference max, p * s_t as
//      fp16 hi + lo into shared memory (B of p . V);
//   5. one barrier; thread 0 issues two tcgen05.mma (m128 n16 k16, one per 16
//      tokens) per group into the accumulators in tensor memory and commits
//      them to an mbarrier that the next round waits on before it overwrites
//      A and B.
// The reference max moves only when a score exceeds it by more than 0.5
// (log2 units), so weights stay <= 2^0.5 and p * s_t fits fp16 for any scale
// (2^0.5 * 43669 < 65504). Step 4 is done speculatively; when some warp sees a
// larger score the barrier says so, every warp takes the new reference,
// rescales its lanes of the accumulators and recomputes its weights.
// The window chunks then run one at a time on the whole block (warp i: tokens
// 8i .. 8i + 7 of q . k^T; every warp: its channels into tensor memory), into
// their own accumulators. Each block writes unnormalized (m, l, o) partials
// per query head; the last block of a pair merges them (finish_split).
// Every wait is bounded: after kWaitLimitNs the block sets bit 0 of the
// status word, stops issuing work, lets what it issued land, contributes
// nothing more and frees its tensor memory.
template <int D, int KB, int VB, class SeqT>
__global__ void __launch_bounds__(128, 4) kivi_decode_tc_kernel(KiviDecodeArgs a, SeqT seqs) {
  using P = Kivi<D, KB, VB>;
  using S = TcSmem<D, KB, VB>;
  constexpr int NS = S::NS;
  constexpr bool kPaged = !std::is_same<SeqT, NoSeqs>::value;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bsm = smem;               // B of p . V: two buffers of 4 group slots
  uint8_t* area = smem + S::B_BYTES;  // ring of record stages / window rows / output rows
  const uint32_t bsm_s = smem_addr(bsm), area_s = smem_addr(area);
  __shared__ __align__(8) uint64_t tma_bar[NS];
  __shared__ __align__(8) uint64_t mma_bar[2];
  __shared__ __align__(8) uint64_t win_bar;
  __shared__ uint32_t tmem_s;
  __shared__ float mx_s[4][8];     // per-warp round maxima of each query head
  __shared__ float lz_s[4][8][2];  // per-warp sum p and sum p z
  __shared__ float ml_s[2][8];     // the block's partial: m, l per query head
  __shared__ int abort_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int gq = a.q_heads / a.kv_heads;

  if (warp == 0) {
    tmem_alloc(&tmem_s, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(&tma_bar[i], 1);
    mbar_init(&mma_bar[0], 1);
    mbar_init(&mma_bar[1], 1);
    mbar_init(&win_bar, 1);
    fence_mbar_init();
  }
  if (tid == 64) abort_s = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes
  const int ch = warp * 32 + lane;                                        // the channel of this lane
  const bool has_ch = (D == 128) || warp * 32 < D;  // D = 64: warps 0-1 hold the channels
  constexpr uint32_t kIdesc = tc_idesc_f16_f32<128, 16>();

  // Counters every thread keeps identically.
  uint32_t n_commit = 0;   // MMA commits issued (commit k arrives on mma_bar[k & 1])
  uint32_t ring_next = 0;  // ring uses issued (use u: stage u % NS, phase (u / NS) & 1)
  uint32_t ring_done = 0;  // ring uses this thread has seen complete
  uint32_t wphase = 0;     // phase of the window barrier
  bool win_pending = false;
  bool aborted = false;    // a wait gave up: no more work (uniform: set after barriers)

  auto wait_mma = [&]() -> bool {  // every MMA issued so far has completed
    if (n_commit == 0) return true;
    const uint32_t k = n_commit - 1;
    return mbar_wait_bounded(&mma_bar[k & 1], (k >> 1) & 1);
  };

  long long all_units = static_cast<long long>(a.n_pairs) * a.pair_stride;
  if constexpr (kPaged) all_units = seqs.unit0[seqs.n_seqs];
  const long long u0 = static_cast<long long>(blockIdx.x) * a.units_per_block;
  const long long u1 = min(all_units, u0 + a.units_per_block);
  for (long long u = u0; u < u1;) {
    int pair, upp, n_grp, n_res;
    long long pbase;
    if constexpr (kPaged) {
      const int sb = seq_of(seqs.unit0, seqs.n_seqs, u);
      n_grp = seqs.n_groups[sb];
      n_res = seqs.n_resid[sb];
      upp = n_grp + kChunkUnits * ((n_res + kGroup - 1) / kGroup);
      // each pair's range opens with pair_lead units of no work (the cost of
      // one more segment); pbase is its first unit of work
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
    // the previous segment's epilogue is done with the area and the B slots
    fence_proxy_async_smem();
    __syncthreads();

    const int n_chunks = (n_res + kGroup - 1) / kGroup;
    const int g_begin = min(n_grp, lo);
    const int g_end = min(n_grp, hi);
    const int c_begin = min(n_chunks, max(0, lo - n_grp + kChunkUnits - 1) / kChunkUnits);
    const int c_end = min(n_chunks, max(0, hi - n_grp + kChunkUnits - 1) / kChunkUnits);
    const int n_here = g_end - g_begin;
    const int n_rounds = aborted ? 0 : (n_here + 3) / 4;

    // contiguous: the pair's records, groups one after the other
    const long long rec0 = bh * a.groups_cap;
    const uint8_t* kc_g = a.k_codes + rec0 * P::KC;
    const uint8_t* km_g = a.k_meta + rec0 * P::KM;
    const uint8_t* vc_g = a.v_codes + rec0 * P::VC;
    const uint8_t* vm_g = a.v_meta + rec0 * P::VM;
    // paged: lane l of warp 1 holds the pool block of group g_begin + tbase + l
    TableLanes<kPaged> tl;
    auto load_table = [&](int base) {  // warp 1, warp-wide
      if constexpr (kPaged) {
        tl.tbase = base;
        const int grp = g_begin + base + lane;
        if (grp < g_end)
          tl.tblk = min(max(__ldg(seqs.pools.block_table + static_cast<long long>(b) * a.groups_cap + grp), 0),
                        seqs.pools.num_blocks - 1);
      }
    };
    const uint32_t rb = ring_next;  // ring use of this segment's round 0
    // round k's records into stage (rb + k) % NS (warp 1, warp-wide; lane 0 issues)
    auto issue_round = [&](int k) {
      const uint32_t use = rb + k;
      uint8_t* dst = area + (use % NS) * S::ROUND;
      uint64_t* bb = &tma_bar[use % NS];
      const int grp = g_begin + 4 * k;
      const int cnt = min(4, g_end - grp);
      if constexpr (kPaged) {
        if (4 * k + 4 > tl.tbase + 32) load_table(4 * k);
        int blk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) blk[i] = __shfl_sync(0xffffffffu, tl.tblk, (4 * k + i - tl.tbase) & 31);
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bb, static_cast<uint32_t>(cnt * P::STAGE));
          const uint8_t* pool_h = a.k_codes + static_cast<long long>(h) * P::STAGE;
          for (int i = 0; i < cnt; ++i)
            bulk_g2s(dst + i * P::STAGE, pool_h + static_cast<long long>(blk[i]) * a.kv_heads * P::STAGE, P::STAGE,
                     bb);
        }
      } else if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bb, static_cast<uint32_t>(cnt * P::STAGE));
        bulk_g2s(dst, kc_g + grp * static_cast<long long>(P::KC), cnt * P::KC, bb);
        bulk_g2s(dst + 4 * P::KC, km_g + grp * static_cast<long long>(P::KM), cnt * P::KM, bb);
        bulk_g2s(dst + 4 * (P::KC + P::KM), vc_g + grp * static_cast<long long>(P::VC), cnt * P::VC, bb);
        bulk_g2s(dst + 4 * (P::KC + P::KM + P::VC), vm_g + grp * static_cast<long long>(P::VM), cnt * P::VM, bb);
      }
    };
    // shared addresses of the records of group slot i of the stage at st
    auto kc_of = [&](uint32_t st, int i) -> uint32_t {
      if constexpr (kPaged) return st + i * P::STAGE;
      else return st + i * P::KC;
    };
    auto km_of = [&](uint32_t st, int i) -> uint32_t {
      if constexpr (kPaged) return st + i * P::STAGE + P::KC;
      else return st + 4 * P::KC + i * P::KM;
    };
    auto vc_of = [&](uint32_t st, int i) -> uint32_t {
      if constexpr (kPaged) return st + i * P::STAGE + P::KC + P::KM;
      else return st + 4 * (P::KC + P::KM) + i * P::VC;
    };
    auto vm_of = [&](uint32_t st, int i) -> uint32_t {
      if constexpr (kPaged) return st + i * P::STAGE + P::KC + P::KM + P::VC;
      else return st + 4 * (P::KC + P::KM + P::VC) + i * P::VM;
    };

    const int n_pre = min(NS, n_rounds);
    if (warp == 1)
      for (int k = 0; k < n_pre; ++k) issue_round(k);
    ring_next += n_pre;

    // accumulators of this segment start at zero (the previous segment's
    // MMAs completed before its epilogue read them)
    if (has_ch) {
      const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      tmem_st16(trow + kColD6, z);
      tmem_st16(trow + kColD8, z);
      tmem_st16(trow + kColDW, z);
      tmem_wait_st();
    }

    // Query fragments of row g (query head h*gq + g), scaled by 2^-e so that
    // |q| < 1 and q * s stays inside the fp16 range.
    const bool row_ok = g < gq;
    const __half* qrow = reinterpret_cast<const __half*>(a.q) +
                         (static_cast<long long>(b) * a.q_heads + h * gq + (row_ok ? g : 0)) * D;
    float2 qv[P::KS][2];
    float qmax = 0.0f;
#pragma unroll
    for (int ks = 0; ks < P::KS; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __half2 v = row_ok ? *reinterpret_cast<const __half2*>(qrow + 16 * ks + 8 * j + 2 * tig)
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
    const float p2e = ldexpf(1.0f, e) * a.scale_log2;
    const float mult6 = kInvP6 * p2e, mult8 = kInvP8 * p2e;

    // q . k_hat of the 32 tokens of one group: 8 scores (log2 units) of this
    // thread's row, tokens 8*nt + 2*tig + {0, 1}.
    auto qk_scores = [&](uint32_t kc, uint32_t km, float (&sc)[8]) {
      uint32_t kw[P::KW];
#pragma unroll
      for (int c = 0; c < P::KW / 4; ++c) {
        const uint4 x = lds128(kc + (c * 32 + lane) * 16);
        kw[4 * c] = x.x;
        kw[4 * c + 1] = x.y;
        kw[4 * c + 2] = x.z;
        kw[4 * c + 3] = x.w;
      }
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
      // q . z on the same tensor pipe, two m16n8k8 per k-step with A = (q of
      // channels 16ks + 2tig.., q of channels 16ks + 8 + 2tig..) as held and B
      // = the zero points of the first (bz0) or second (bz1) 8 channels in
      // every column: row g of bz0 and row g + 8 of bz1 each hold their half
      // of sum_d q_{g,d} z_d (exact fp16 products, fp32 sums), in this
      // thread's row without a shuffle.
      float bz0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, bz1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int ks = 0; ks < P::KS; ++ks) {
        // {s(d0,d0+1), s(d0+8,d0+9), z(d0,d0+1), z(d0+8,d0+9)}
        const uint4 md = lds128(km + (ks * 4 + tig) * 16);
        const __half2 q0 = bits_h2(qs[ks][0]), q1 = bits_h2(qs[ks][1]);
        const __half2 hi0 = __hmul2(q0, bits_h2(md.x));
        const __half2 lo0 = __hfma2(q0, bits_h2(md.x), __hneg2(hi0));
        const __half2 hi1 = __hmul2(q1, bits_h2(md.y));
        const __half2 lo1 = __hfma2(q1, bits_h2(md.y), __hneg2(hi1));
        const uint32_t A0 = h2_bits(hi0), A1 = h2_bits(lo0), A2 = h2_bits(hi1), A3 = h2_bits(lo1);
        mma1688(bz0, qs[ks][0], qs[ks][1], md.z);
        mma1688(bz1, qs[ks][0], qs[ks][1], md.w);
        if constexpr (KB == 2) {
          const uint32_t w = kw[ks];
          const uint32_t l4 = w << 4, r4 = w >> 4, sw = __byte_perm(w, 0u, 0x2301u);
          mma16816(sacc[0], A0, A1, A2, A3, l4 & kMaskP6, r4 & kMaskP6);
          mma16816(sacc[1], A0, A1, A2, A3, l4 & kMaskP8, r4 & kMaskP8);
          mma16816(sacc[2], A0, A1, A2, A3, w & kMaskP6, sw & kMaskP6);
          mma16816(sacc[3], A0, A1, A2, A3, w & kMaskP8, sw & kMaskP8);
        } else {
          const uint32_t w0 = kw[2 * ks], w1 = kw[2 * ks + 1];
          mma16816(sacc[0], A0, A1, A2, A3, (w0 << 6) & kMask4, (w1 << 6) & kMask4);
          mma16816(sacc[1], A0, A1, A2, A3, (w0 << 2) & kMask4, (w1 << 2) & kMask4);
          mma16816(sacc[2], A0, A1, A2, A3, (w0 >> 2) & kMask4, (w1 >> 2) & kMask4);
          mma16816(sacc[3], A0, A1, A2, A3, (w0 >> 6) & kMask4, (w1 >> 6) & kMask4);
        }
      }
      const float bias = (bz0[0] + bz1[2]) * p2e;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float mult = (KB == 2 && (nt & 1)) ? mult8 : mult6;
        sc[2 * nt] = fmaf(sacc[nt][0] + sacc[nt][2], mult, bias);
        sc[2 * nt + 1] = fmaf(sacc[nt][1] + sacc[nt][3], mult, bias);
      }
    };

    float m_ref = -INFINITY, l_run = 0.0f, vz_run = 0.0f;  // head g
    bool first = true;  // no reference yet: nothing to rescale
    // After a barrier that reported a larger score: the new reference of every
    // head (the same in every warp), the accumulators rescaled.
    auto rebase = [&]() {
      const float M = fmaxf(fmaxf(mx_s[0][g], mx_s[1][g]), fmaxf(mx_s[2][g], mx_s[3][g]));
      const float m_new = (M > m_ref + 0.5f) ? M : m_ref;
      const float alpha = fast_exp2(m_ref - m_new);  // 0 from -inf, 1 when unchanged
      const bool moved = __any_sync(0xffffffffu, m_new != m_ref);
      if (!first && moved && has_ch) {
        float al[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) al[q] = __shfl_sync(0xffffffffu, alpha, 4 * q);
        const uint32_t cols[3] = {kColD6, kColD8, kColDW};
#pragma unroll
        for (int rg = 0; rg < 3; ++rg) {
          uint32_t v[16];
          tmem_ld16(trow + cols[rg], v);
          tmem_wait_ld();
#pragma unroll
          for (int n = 0; n < 16; ++n) v[n] = __float_as_uint(__uint_as_float(v[n]) * al[n & 7]);
          tmem_st16(trow + cols[rg], v);
        }
        tmem_wait_st();
      }
      l_run *= alpha;
      vz_run *= alpha;
      m_ref = m_new;
    };

    // ------------------------------- grouped region -------------------------------
    // The value codes of group slot i of the stage at st into A slot i (this
    // warp's 32 channels); the first cnt slots (all four when full).
    const uint32_t ch_off = ch * (4 * VB);  // this lane's channel inside a value-code record
    auto fill_round = [&](uint32_t st, int cnt) {
      if (cnt == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) fill_value_codes<VB>(vc_of(st, i) + ch_off, trow + kColA + 16 * i);
      } else {
        for (int i = 0; i < cnt; ++i) fill_value_codes<VB>(vc_of(st, i) + ch_off, trow + kColA + 16 * i);
      }
    };
    // thread 0: two MMAs per group of the round (16 tokens each) from B buffer bb
    auto issue_pv = [&](uint32_t bb, int cnt) {
      const uint64_t d0 = smem_desc_kmajor(bb, kLbo, kSbo);  // + (bytes >> 4) moves the start address
      if (cnt == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tc_mma_f16_tmem_a(tmem + kColD6, tmem + kColA + 16 * i, d0 + ((i * kBSlot) >> 4), kIdesc, 1u);
          tc_mma_f16_tmem_a(tmem + (VB == 2 ? kColD8 : kColD6), tmem + kColA + 16 * i + 8,
                            d0 + ((i * kBSlot + 256) >> 4), kIdesc, 1u);
        }
      } else {
        for (int i = 0; i < cnt; ++i) {
          tc_mma_f16_tmem_a(tmem + kColD6, tmem + kColA + 16 * i, d0 + ((i * kBSlot) >> 4), kIdesc, 1u);
          tc_mma_f16_tmem_a(tmem + (VB == 2 ? kColD8 : kColD6), tmem + kColA + 16 * i + 8,
                            d0 + ((i * kBSlot + 256) >> 4), kIdesc, 1u);
        }
      }
    };
    for (int r = 0; r < n_rounds; ++r) {
      const uint32_t use = rb + r;
      const uint32_t st = area_s + (use % NS) * S::ROUND;
      const int cnt = min(4, n_here - 4 * r);
      // B of this batch: the buffer the batch before last read (its MMAs are known complete)
      const uint32_t bbuf = bsm_s + (n_commit & 1) * (4 * kBSlot);
      const uint32_t brow = bbuf + warp * kBSlot + g * 16 + tig * 4;
      bool ok = mbar_wait_bounded(&tma_bar[use % NS], (use / NS) & 1);
      if (ok) ring_done = use + 1;
      float sc[8];
      if (warp < cnt) {
        qk_scores(kc_of(st, warp), km_of(st, warp), sc);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = -INFINITY;
      }
      float mx = sc[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) mx = fmaxf(mx, sc[i]);
      mx = quad_max(mx);
      const bool need = mx > m_ref + 0.5f;
      if (tig == 0) mx_s[warp][g] = mx;
      const bool wneed = __any_sync(0xffffffffu, need);
      float lsum = 0.0f, vzsum = 0.0f;
      if (!wneed && warp < cnt) group_weights(sc, m_ref, vm_of(st, warp), brow, tig, lsum, vzsum);
      ok = wait_mma() && ok;  // the previous batch's MMAs have read A
      tc_fence_after();
      if (has_ch) fill_round(st, cnt);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      if (!ok) {
        abort_s = 1;
        report_timeout(a.status);
      }
      if (__syncthreads_or(need || !ok)) {
        if (abort_s) {
          aborted = true;
          break;
        }
        tc_fence_after();
        rebase();
        lsum = vzsum = 0.0f;
        if (warp < cnt) group_weights(sc, m_ref, vm_of(st, warp), brow, tig, lsum, vzsum);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
      }
      first = false;
      l_run += lsum;
      vz_run += vzsum;
      if (tid == 0) {
        tc_fence_after();
        issue_pv(bbuf, cnt);
        tc_commit(&mma_bar[n_commit & 1]);
      }
      ++n_commit;
      if (r + NS < n_rounds) {
        if (warp == 1) issue_round(r + NS);  // into the stage this round has left
        ++ring_next;
      }
    }

    // ------------------------ fp16 window, 32-token chunks ------------------------
    for (int c = c_begin; c < c_end && !aborted; ++c) {
      if (c == c_begin) asm volatile("griddepcontrol.wait;" ::: "memory");  // the window is complete
      const int t0 = c * kGroup;
      const int nv = min(kGroup, n_res - t0);
      uint8_t* kwin = area;
      uint8_t* vwin = area + 32 * S::WIN_ROW;
      const long long row0 = bh * a.res_cap + t0;
      if (warp == 1) {
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(&win_bar, static_cast<uint32_t>(2 * nv * D * 2));
        __syncwarp();
        if (lane < nv) {
          bulk_g2s(kwin + lane * S::WIN_ROW, a.k_res + (row0 + lane) * D, D * 2, &win_bar);
          bulk_g2s(vwin + lane * S::WIN_ROW, a.v_res + (row0 + lane) * D, D * 2, &win_bar);
        }
      }
      win_pending = true;
      bool ok = mbar_wait_bounded(&win_bar, wphase);
      if (ok) {
        wphase ^= 1u;
        win_pending = false;
      }
      // q . k^T of tokens 8*warp .. +7 (A = q, rows 8-15 zero; B = key rows)
      float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int ks = 0; ks < P::KS; ks += 2) {
        uint32_t kb[4];
        ldsm_x4(kb, kwin + (8 * warp + (lane & 7)) * S::WIN_ROW + (16 * ks + 8 * (lane >> 3)) * 2);
        mma16816(sacc, qs[ks][0], 0u, qs[ks][1], 0u, kb[0], kb[1]);
        mma16816(sacc, qs[ks + 1][0], 0u, qs[ks + 1][1], 0u, kb[2], kb[3]);
      }
      float sc[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) sc[i] = (8 * warp + 2 * tig + i < nv) ? sacc[i] * p2e : -INFINITY;
      const float mx = quad_max(fmaxf(sc[0], sc[1]));
      const bool need = mx > m_ref + 0.5f;
      if (tig == 0) mx_s[warp][g] = mx;
      const bool wneed = __any_sync(0xffffffffu, need);
      ok = wait_mma() && ok;
      tc_fence_after();
      uint8_t* bbuf = bsm + (n_commit & 1) * (4 * kBSlot);
      float lsum = 0.0f;
      if (!wneed) window_weights(sc, m_ref, bbuf, warp, g, tig, lsum);
      if (has_ch) fill_window_values(vwin, S::WIN_ROW, nv, ch, trow + kColA);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      if (!ok) {
        abort_s = 1;
        report_timeout(a.status);
      }
      if (__syncthreads_or(need || !ok)) {
        if (abort_s) {
          aborted = true;
          break;
        }
        tc_fence_after();
        rebase();
        lsum = 0.0f;
        window_weights(sc, m_ref, bbuf, warp, g, tig, lsum);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
      }
      first = false;
      l_run += lsum;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t bb = smem_addr(bbuf);
        tc_mma_f16_tmem_a(tmem + kColDW, tmem + kColA, smem_desc_kmajor(bb, kLbo, kSbo), kIdesc, 1u);
        tc_mma_f16_tmem_a(tmem + kColDW, tmem + kColA + 8, smem_desc_kmajor(bb + 256, kLbo, kSbo), kIdesc, 1u);
        tc_commit(&mma_bar[n_commit & 1]);
      }
      ++n_commit;
    }

    // ------------------------------- segment partial -------------------------------
    const bool ok_end = aborted || wait_mma();
    if (!ok_end) {
      abort_s = 1;
      report_timeout(a.status);
    }
    if (__syncthreads_or(!ok_end)) aborted = true;
    const bool dead = aborted;
    tc_fence_after();
    l_run = quad_sum(l_run);
    vz_run = quad_sum(vz_run);
    if (tig == 0) {
      lz_s[warp][g][0] = dead ? 0.0f : l_run;
      lz_s[warp][g][1] = dead ? 0.0f : vz_run;
      if (warp == 0) ml_s[0][g] = dead ? -INFINITY : m_ref;
    }
    __syncthreads();
    float* o_s = reinterpret_cast<float*>(area);  // [8 rows][D]
    if (has_ch) {
      uint32_t d6[16], d8[16], dw[16];
      tmem_ld16(trow + kColD6, d6);
      tmem_ld16(trow + kColD8, d8);
      tmem_ld16(trow + kColDW, dw);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float vz = (lz_s[0][q][1] + lz_s[1][q][1]) + (lz_s[2][q][1] + lz_s[3][q][1]);
        const float w6 = __uint_as_float(d6[q]) + __uint_as_float(d6[q + 8]);
        const float w8 = __uint_as_float(d8[q]) + __uint_as_float(d8[q + 8]);
        const float ww = __uint_as_float(dw[q]) + __uint_as_float(dw[q + 8]);
        const float o = fmaf(w6, kInvP6, fmaf(w8, kInvP8, ww + vz));
        o_s[q * D + ch] = dead ? 0.0f : o;
      }
    }
    if (tid < 8) ml_s[1][tid] = (lz_s[0][tid][0] + lz_s[1][tid][0]) + (lz_s[2][tid][0] + lz_s[3][tid][0]);
    // the kernel before this one has finished before any workspace write (see tc_dispatch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    finish_split<D, 1>(o_s, ml_s[0], ml_s[1], gq, static_cast<long long>(b) * a.q_heads + h * gq, split, n_splits,
                       a.part_stride, a.part_o, a.part_ml, a.counters + bh, a.out, a.out_fp32);
  }

  // Let every copy and MMA this block issued land, then free its tensor memory.
  if (aborted) {
    for (uint32_t x = ring_done; x < ring_next; ++x) (void)mbar_wait_bounded(&tma_bar[x % NS], (x / NS) & 1);
    if (win_pending) (void)mbar_wait_bounded(&win_bar, wphase);
  }
  (void)wait_mma();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Resident blocks per SM from the block's registers and shared memory and the
// tensor-memory columns it allocates. (The runtime's occupancy calculator
// answers 1 for any kernel that allocates tensor memory, as if each block
// could take all 512 columns; this kernel takes kTmemCols.)
template <int D, int KB, int VB, class SeqT>
int tc_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    constexpr int smem = TcSmem<D, KB, VB>::BYTES;
    auto kern = kivi_decode_tc_kernel<D, KB, VB, SeqT>;
    cudaFuncAttributes fa{};
    int regs_sm = 0, smem_sm = 0, smem_rsv = 0, threads_sm = 0;
    int n = 1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
        cudaFuncGetAttributes(&fa, kern) == cudaSuccess &&
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) == cudaSuccess) {
      const int regs_block = ((fa.numRegs + 7) / 8) * 8 * 128;  // allocated per warp in steps of 8 per thread
      const int smem_block = static_cast<int>(fa.sharedSizeBytes) + smem + smem_rsv;
      n = kTmemBlocksPerSm;
      if (regs_block > 0) n = n < regs_sm / regs_block ? n : regs_sm / regs_block;
      if (smem_block > 0) n = n < smem_sm / smem_block ? n : smem_sm / smem_block;
      n = n < threads_sm / 128 ? n : threads_sm / 128;
      if (n < 1) n = 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// The decode is launched as a programmatic dependent of the kernel before it
// on the stream. Only the token copy of kv_append_token (and of the window
// fill) lets its dependent start early; every other kernel releases it at its
// end as usual. So the decode's grouped rounds, which read only group records
// and q (complete before that copy started), overlap the copy, while the fp16
// window and the workspace (partials, split counters, shared with the
// previous decode) are touched only after griddepcontrol.wait, i.e. after the
// preceding kernel has completed.
template <int D, int KB, int VB, class SeqT>
cudaError_t tc_dispatch(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  constexpr int smem = TcSmem<D, KB, VB>::BYTES;
  auto kern = kivi_decode_tc_kernel<D, KB, VB, SeqT>;
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
cudaError_t tc_by_key(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  switch (a.head_dim * 100 + a.k_bits * 10 + a.v_bits) {
    case 6422: return tc_dispatch<64, 2, 2>(a, seqs, s);
    case 6424: return tc_dispatch<64, 2, 4>(a, seqs, s);
    case 6442: return tc_dispatch<64, 4, 2>(a, seqs, s);
    case 6444: return tc_dispatch<64, 4, 4>(a, seqs, s);
    case 12822: return tc_dispatch<128, 2, 2>(a, seqs, s);
    case 12824: return tc_dispatch<128, 2, 4>(a, seqs, s);
    case 12842: return tc_dispatch<128, 4, 2>(a, seqs, s);
    case 12844: return tc_dispatch<128, 4, 4>(a, seqs, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class SeqT>
int tc_occupancy_by_key(int head_dim, int k_bits, int v_bits) {
  switch (head_dim * 100 + k_bits * 10 + v_bits) {
    case 6422: return tc_occupancy<64, 2, 2, SeqT>();
    case 6424: return tc_occupancy<64, 2, 4, SeqT>();
    case 6442: return tc_occupancy<64, 4, 2, SeqT>();
    case 6444: return tc_occupancy<64, 4, 4, SeqT>();
    case 12822: return tc_occupancy<128, 2, 2, SeqT>();
    case 12824: return tc_occupancy<128, 2, 4, SeqT>();
    case 12842: return tc_occupancy<128, 4, 2, SeqT>();
    case 12844: return tc_occupancy<128, 4, 4, SeqT>();
    default: return 1;
  }
}

}  // namespace

cudaError_t launch_kivi_decode(const KiviDecodeArgs& a, cudaStream_t s) { return tc_by_key(a, NoSeqs{}, s); }

cudaError_t launch_kivi_decode_paged(const KiviDecodeArgs& a, const PagedSeqs& seqs, cudaStream_t s) {
  return tc_by_key(a, seqs, s);
}

int kivi_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return tc_occupancy_by_key<NoSeqs>(head_dim, k_bits, v_bits);
}

int kivi_paged_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return tc_occupancy_by_key<PagedSeqs>(head_dim, k_bits, v_bits);
}

}  // namespace kvq
