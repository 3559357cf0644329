// FP8 paged KV cache kernels for sm_103a (E4M3 or E5M2, one scale per tensor
// or per kv head): amax (two passes, no atomics), scale = amax / FMAX (448 for
// E4M3, 57344 for E5M2), cast + scatter into paged blocks, and split-K decode
// attention over the paged cache.
//
// Method: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 5
// (E4M3 = 1 sign, 4 exponent, 3 mantissa bits); "大模型量化从0到1（十三）：KV Cache
// 量化" (CSDN), section 10 (q = cast_fp8(x / s), x_hat = float(q) * s, per-tensor
// scale) and section 13 (paged blocks through a block table); "LLM推理加速KV Cache
// 量化压缩实战方案" (yunthe), custom-cache section (scale = max|x| / 448); CSDN
// section 10.1 (per-head scales) and section 18.4 (E5M2); section 18.7
// (FP8-domain attention: the query quantized to FP8 as well, q.k^T on FP8
// operands).
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kBlock = 16;  // tokens per paged block

// ---------------------------------------------------------------------------
// amax: max |x| as the maximum of the fp16 magnitude bits (|x| orders like its
// bits; a NaN's bits exceed every finite value's and infinity's).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t max_mag_bits(uint32_t m, const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
  return m;
}

// Per tensor (gridDim.y == 1): the whole [B, H, S, D] tensor, grid-strided.
// Per kv head (gridDim.y == H): block (x, h) strides over head h's B slices of
// row_vecs = S * D / 8 16-byte vectors. Partial (h, x) goes to
// partials[h * gridDim.x + x].
__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint4* __restrict__ x, long long n_vec, int batch,
                                                       int heads, long long row_vecs, uint32_t* __restrict__ partials) {
  uint32_t m = 0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (gridDim.y == 1) {
    long long i = t0;
    for (; i + 3 * stride < n_vec; i += 4 * stride) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(x + i + u * stride);
#pragma unroll
      for (int u = 0; u < 4; ++u) m = max_mag_bits(m, v[u]);
    }
    for (; i < n_vec; i += stride) m = max_mag_bits(m, __ldcs(x + i));
  } else {
    const int h = blockIdx.y;
    for (int b = 0; b < batch; ++b) {
      const uint4* row = x + (static_cast<long long>(b) * heads + h) * row_vecs;
      long long i = t0;
      for (; i + 3 * stride < row_vecs; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(row + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) m = max_mag_bits(m, v[u]);
      }
      for (; i < row_vecs; i += stride) m = max_mag_bits(m, __ldcs(row + i));
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < (blockDim.x >> 5); ++k) r = max(r, wm[k]);
    partials[blockIdx.y * gridDim.x + blockIdx.x] = r;
  }
}

// scale[h] = fl32(amax / FMAX), or 1 when the tensor (or head) is all zeros;
// one block per scale, over its n partials.
__global__ void __launch_bounds__(256) fp8_scale_kernel(const uint32_t* __restrict__ partials, int n, float fmax,
                                                        float* __restrict__ scale) {
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = max(m, partials[blockIdx.x * n + i]);
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < (blockDim.x >> 5); ++k) r = max(r, wm[k]);
    const float amax = __half2float(__ushort_as_half(static_cast<unsigned short>(r)));
    scale[blockIdx.x] = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, fmax);
  }
}

// ---------------------------------------------------------------------------
// Cast + scatter: each warp takes (b, h, logical block) units in turn and
// stages each unit's 16 x D fp16 values in one of its two shared-memory
// buffers with 16-byte asynchronous copies issued one unit ahead, so the
// loads of the next unit are in flight while this one is converted. Every
// lane then writes its D/32 16-byte chunks of the fragment-ordered block
// (chunk c of lane l at byte (c*32 + l)*16, so each store instruction of the
// warp covers 512 contiguous bytes).
// ---------------------------------------------------------------------------
constexpr int kCastWarps = 4;


// x / scale, the IEEE fp32 quotient of the formula. MODE 0: the IEEE division
// itself. MODE 1 and 2: from y = RN(1/scale) and one correction step, which is
// bit-identical for scales in [2^-96, 2^96]; MODE 1 also passes an infinite x
// through (a static scale may meet infinities), MODE 2 leaves that test out: a
// dynamic scale amax / 448 is only that finite when the tensor holds no
// infinity or NaN (either one makes amax, hence the scale, non-finite).
template <int MODE>
__device__ __forceinline__ float scaled(float x, float scale, float y) {
  if constexpr (MODE == 0) {
    (void)y;
    return __fdiv_rn(x, scale);
  } else if constexpr (MODE == 1) {
    return div_rn_by_rcp_signed(x, scale, y);
  } else {
    return copysignf(div_rn_by_rcp(x, scale, y), x);
  }
}

// scaled<MODE> of both halves of an fp16 pair, the reciprocal path in packed
// fp32 operations (the same steps, so the same quotients).
template <int MODE>
__device__ __forceinline__ float2 scaled_pair(uint32_t xh2, float scale, float y) {
  const float2 x = __half22float2(bits_h2(xh2));
  if constexpr (MODE == 0) {
    (void)y;
    return make_float2(__fdiv_rn(x.x, scale), __fdiv_rn(x.y, scale));
  } else {
    const float2 q0 = __fmul2_rn(x, make_float2(y, y));
    const float2 r = __ffma2_rn(q0, make_float2(-scale, -scale), x);
    const float2 q = __ffma2_rn(r, make_float2(y, y), q0);
    float2 o = make_float2(copysignf(q.x, x.x), copysignf(q.y, x.y));
    if constexpr (MODE == 1) {
      if (isinf(x.x)) o.x = x.x;
      if (isinf(x.y)) o.y = x.y;
    }
    return o;
  }
}

// ROLE 2: keys (4-byte words = m16n8k32 B fragments), ROLE 1: values (token
// pairs per channel). Byte pairs of the lane's stream come as fp16 pairs:
// keys two adjacent channels of a token (one 32-bit load), values two tokens of
// a channel (a transposed ldmatrix gives four of them).
template <int D, int MODE, int FMT, int ROLE>
__device__ __forceinline__ void cast_units(const Fp8QuantArgs& a, __half* bufs) {
  constexpr int RS = D + 8;  // padded row stride (halves): rows start 4 banks apart
  constexpr int BUF = kBlock * RS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gg = lane >> 2, tg = lane & 3;
  const int nb = (a.seq_len + kBlock - 1) / kBlock;
  const long long units = static_cast<long long>(a.batch) * a.kv_heads * nb;
  const long long stride = static_cast<long long>(gridDim.x) * kCastWarps;

  // Start staging unit u into buffer k (one commit group per call, empty when
  // the unit is skipped); returns its physical block, or -1 to skip it.
  auto stage = [&](long long u, int k) -> int {
    const int j = static_cast<int>(u % nb);
    const long long bh = u / nb;
    const int b = static_cast<int>(bh / a.kv_heads);
    const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + j];
    if (blk >= 0 && blk < a.num_blocks) {  // uniform per warp: no write outside the pool
      const int t0 = j * kBlock, ntok = min(kBlock, a.seq_len - t0);
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (bh * a.seq_len + t0) * static_cast<long long>(D));
      __half* dst = bufs + k * BUF;
#pragma unroll
      for (int i = lane; i < kBlock * D / 8; i += 32) {
        const int tok = i / (D / 8), c8 = i % (D / 8);
        if (tok < ntok)
          cp_async16(dst + tok * RS + 8 * c8, src + i);
        else
          *reinterpret_cast<uint4*>(dst + tok * RS + 8 * c8) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();
    return (blk >= 0 && blk < a.num_blocks) ? blk : -1;
  };

  long long u = static_cast<long long>(blockIdx.x) * kCastWarps + warp;
  int k = 0;
  int blk_of[2] = {-1, -1};
  if (u < units) blk_of[0] = stage(u, 0);
  for (; u < units; u += stride, k ^= 1) {
    // the other buffer was read in the previous iteration (ended with a __syncwarp)
    if (u + stride < units)
      blk_of[k ^ 1] = stage(u + stride, k ^ 1);
    else
      cp_async_commit();
    cp_async_wait_all_but_newest();
    __syncwarp();  // every lane's copies of this unit have landed
    const int blk = blk_of[k];
    if (blk >= 0) {
      const __half* xs = bufs + k * BUF;
      const int j = static_cast<int>(u % nb);
      const int h = static_cast<int>((u / nb) % a.kv_heads);
      const int ntok = min(kBlock, a.seq_len - j * kBlock);
      const float scale = a.scale[a.per_head ? h : 0];
      const float y = (MODE == 0) ? 0.0f : __frcp_rn(scale);
      uint4* dst = reinterpret_cast<uint4*>(a.pool + (static_cast<long long>(blk) * a.kv_heads + h) * (kBlock * D));
      const bool full = ntok == kBlock;  // else rows past the sequence are zeroed bytes
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t pr[8];  // byte pair kk of the lane's 16-byte chunk c (pair index 8c + kk of its stream)
        if constexpr (ROLE == 2) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 4-byte word w = (nt * (D/32) + k2) * 2 + r: channels 32k2 + 16r + 4tg .. +3 of token 8nt + gg
            const int i = 8 * c + kk, w = i >> 1, nt = w / (D / 16), rem = w % (D / 16), k2 = rem >> 1, r = rem & 1;
            const int tok = 8 * nt + gg, ch = 32 * k2 + 16 * r + 4 * tg + 2 * (i & 1);
            const float2 q = scaled_pair<MODE>(*reinterpret_cast<const uint32_t*>(xs + tok * RS + ch), scale, y);
            pr[kk] = f32x2_to_fp8x2<FMT>(q.x, q.y);
            if (!full && tok >= ntok) pr[kk] = 0u;
          }
        } else {
          // pair i = 2nt + r: tokens 8r + 2tg, +1 of channel 8nt + gg (nt = 4c + e for tile e)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            uint32_t t4[4];
            ldsm_x4_trans(t4, xs + (8 * r + (lane & 7)) * RS + 8 * (4 * c + (lane >> 3)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 q = scaled_pair<MODE>(t4[e], scale, y);
              uint32_t v = f32x2_to_fp8x2<FMT>(q.x, q.y);
              const int t0 = 8 * r + 2 * tg;
              if (!full) v &= (t0 < ntok ? 0x00FFu : 0u) | (t0 + 1 < ntok ? 0xFF00u : 0u);
              pr[2 * e + r] = v;
            }
          }
        }
        dst[c * 32 + lane] = make_uint4(pr[0] | (pr[1] << 16), pr[2] | (pr[3] << 16), pr[4] | (pr[5] << 16),
                                        pr[6] | (pr[7] << 16));
      }
    }
    __syncwarp();  // this buffer is refilled next iteration
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int D, int FMT>
__global__ void __launch_bounds__(32 * kCastWarps) fp8_cast_kernel(Fp8QuantArgs a) {
  __shared__ __align__(16) __half bufs[kCastWarps][2 * kBlock * (D + 8)];
  __half* mine = bufs[threadIdx.x >> 5];
  // the reciprocal path when every scale is in its exact range (the same decision for the whole grid)
  bool fast = true;
  for (int h = 0; h < (a.per_head ? a.kv_heads : 1); ++h) fast &= (a.scale[h] >= 0x1p-96f && a.scale[h] <= 0x1p96f);
  const int mode = !fast ? 0 : (a.static_scale ? 1 : 2);
  if (a.value_layout == 2) {
    if (mode == 0) cast_units<D, 0, FMT, 2>(a, mine);
    else if (mode == 1) cast_units<D, 1, FMT, 2>(a, mine);
    else cast_units<D, 2, FMT, 2>(a, mine);
  } else {
    if (mode == 0) cast_units<D, 0, FMT, 1>(a, mine);
    else if (mode == 1) cast_units<D, 1, FMT, 1>(a, mine);
    else cast_units<D, 2, FMT, 1>(a, mine);
  }
}

// ---------------------------------------------------------------------------
// The query in E4M3 (FP8-domain attention): after fp8_amax_kernel's per-block
// partials over q, every block of the cast reduces the partials itself
// (q_scale = fl32(amax / 448), 1 for an all-zero q; block 0 stores it), then
// casts 8 values per thread and step by the same quotient as the cache cast,
// row-major bytes out. Two launches: a one-block query pass (one SM reads
// ~35 GB/s) and a separate scale kernel both cost more.
// ---------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ void cast_query(const Fp8QueryArgs& a, float scale) {
  const float y = (MODE == 0) ? 0.0f : __frcp_rn(scale);
  const long long n_vec = a.n / 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_vec;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(a.q)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(bits_h2(w[k]));
      const uint32_t pair = f32x2_to_fp8x2<0>(scaled<MODE>(f.x, scale, y), scaled<MODE>(f.y, scale, y));
      if (k & 1)
        out[k >> 1] |= pair << 16;
      else
        out[k >> 1] = pair;
    }
    reinterpret_cast<uint2*>(a.q8)[i] = make_uint2(out[0], out[1]);
  }
}

__global__ void __launch_bounds__(256) fp8_query_cast_kernel(Fp8QueryArgs a) {
  uint32_t m = 0;
  for (int i = threadIdx.x; i < a.amax_blocks; i += blockDim.x) m = max(m, a.partials[i]);
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t wm[8];
  __shared__ float s_scale;
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < 8; ++k) r = max(r, wm[k]);
    const float amax = __half2float(__ushort_as_half(static_cast<unsigned short>(r)));
    const float scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    s_scale = scale;
    if (blockIdx.x == 0) *a.q_scale = scale;
  }
  __syncthreads();
  const float scale = s_scale;
  if (scale >= 0x1p-96f && scale <= 0x1p96f)
    cast_query<2>(a, scale);
  else
    cast_query<0>(a, scale);
}

// ---------------------------------------------------------------------------
// Split-K decode attention over the paged FP8 cache.
// Grid (splits, H_kv, B), 4 warps; warp w of block x takes logical blocks
// x*bps + w, x*bps + w + 4, ... through a ring of STAGES stages (K block and
// V block of one kv head, 16*D bytes each) filled by bulk copies.
//   q.k^T : A = q (fp16, exact, channels permuted as the keys' order), B =
//           FP8 keys converted to fp16 (exact);
//           with QF (FP8-domain attention) A = the E4M3 query bytes and B =
//           the key bytes as stored (the keys' order is the m16n8k32 one), on the FP8 tensor path
//           (m16n8k32), scores scaled by q_scale * k_scale.
//   p.V   : A = p split into fp16 hi + lo rows, B = E4M3 values as fp16.
// ---------------------------------------------------------------------------
template <int D, int STAGES>
struct Fp8Smem {
  static constexpr int BAR_BYTES = 128;
  static constexpr int STAGE = 2 * kBlock * D;
  static constexpr int RING = 4 * STAGES * STAGE;
  static constexpr int COMBINE = (4 * 8 * D + 64) * 4;
  static constexpr int AREA = RING > COMBINE ? RING : COMBINE;
  static constexpr int BYTES = BAR_BYTES + AREA;
};

// The two fp16x2 operands of one word of four FP8 bytes: bytes 0-1 and bytes
// 2-3. An E5M2 byte is the top byte of the fp16 of the same value, so each
// half is one byte permute straight from the word (no extraction of the 16-bit
// half first); E4M3 converts each 16-bit half with its conversion instruction.
template <int FMT>
__device__ __forceinline__ uint32_t fp8_lo_pair(uint32_t w) {
  if constexpr (FMT == 1)
    return __byte_perm(w, 0u, 0x1404u);
  else
    return fp8x2_to_f16x2<FMT>(static_cast<uint16_t>(w & 0xFFFFu));
}
template <int FMT>
__device__ __forceinline__ uint32_t fp8_hi_pair(uint32_t w) {
  if constexpr (FMT == 1)
    return __byte_perm(w, 0u, 0x3424u);
  else
    return fp8x2_to_f16x2<FMT>(static_cast<uint16_t>(w >> 16));
}

// d += A (16 x 32 E4M3, rows g / g + 8) * B (32 x 8, E4M3 or E5M2 per FMT), f32.
template <int FMT>
__device__ __forceinline__ void mma_fp8_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  if constexpr (FMT == 0) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e5m2.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <int D, int STAGES, int FMT, bool QF>
__global__ void __launch_bounds__(128) fp8_decode_kernel(Fp8DecodeArgs a) {
  using S = Fp8Smem<D, STAGES>;
  constexpr int KS = D / 16, NT = D / 8, CH = D / 32;  // CH: 16-byte chunks per lane
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* area = smem + S::BAR_BYTES;
  float* o_s = reinterpret_cast<float*>(area);
  float* m_s = o_s + 4 * 8 * D;
  float* l_s = m_s + 32;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int gq = a.q_heads / a.kv_heads;
  const int len = min(max(a.seq_lens[b], 0), a.max_blocks * kBlock);
  const int nblk = (len + kBlock - 1) / kBlock;
  const int j_begin = split * a.blocks_per_split;
  const int j_end = min(nblk, j_begin + a.blocks_per_split);
  const int n_here = j_end - j_begin;
  const int n_mine = (n_here > warp) ? (n_here - warp + 3) / 4 : 0;
  uint64_t* bar = bars + warp * STAGES;
  uint8_t* ring = area + warp * STAGES * S::STAGE;
  const int32_t* table = a.block_table + static_cast<long long>(b) * a.max_blocks;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // Physical block of the warp's j-th logical block; out-of-range table
  // entries are clamped so that a bad table cannot address outside the pool.
  auto phys = [&](int j) -> long long {
    const int blk = table[j_begin + warp + 4 * j];
    return static_cast<long long>(min(max(blk, 0), a.num_blocks - 1));
  };
  auto issue = [&](int j, long long blk) {
    const long long off = (blk * a.kv_heads + h) * (kBlock * D);
    uint8_t* dst = ring + (j % STAGES) * S::STAGE;
    uint64_t* bb = &bar[j % STAGES];
    mbar_arrive_expect_tx(bb, S::STAGE);
    bulk_g2s(dst, a.k_pool + off, kBlock * D, bb);
    bulk_g2s(dst + kBlock * D, a.v_pool + off, kBlock * D, bb);
  };
  if (lane == 0) {
    for (int j = 0; j < STAGES && j < n_mine; ++j) issue(j, phys(j));
  }

  const bool row_ok = g < gq;
  const __half* qrow = reinterpret_cast<const __half*>(a.q) +
                       (static_cast<long long>(b) * a.q_heads + h * gq + (row_ok ? g : 0)) * D;
  // fp16 query: A fragments of m16n8k16 (rows g, channels 16ks + 8jj + 2tig, +1);
  // E4M3 query (QF): A fragments of m16n8k32 (rows g, channels 32kk + 16jj + 4tig .. +3)
  constexpr int QW = QF ? D / 32 : KS;
  uint32_t qa[QW][2];
  if constexpr (QF) {
    const uint8_t* q8row = a.q8 + (static_cast<long long>(b) * a.q_heads + h * gq + (row_ok ? g : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < QW; ++kk)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
        qa[kk][jj] = row_ok ? *reinterpret_cast<const uint32_t*>(q8row + 32 * kk + 16 * jj + 4 * tig) : 0u;
  } else {
    // The keys are stored in the m16n8k32 order (4 consecutive channels
    // 16ks + 4tig .. +3 per word). A dot product does not depend on the order
    // of its terms, so k-step ks pairs its K rows with channels permuted
    // alike on both sides: rows 2tig, 2tig + 1 <-> channels 16ks + 4tig, +1
    // (b0 = bytes 0-1 of the word, a0), rows 2tig + 8, + 9 <-> channels
    // 16ks + 4tig + 2, + 3 (b1 = bytes 2-3, a2).
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
        qa[ks][jj] = row_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 4 * tig + 2 * jj) : 0u;
  }
  const float kmul = a.k_scale[a.per_head ? h : 0] * a.scale_log2 * (QF ? *a.q_scale : 1.0f);
  const float vscale = a.v_scale[a.per_head ? h : 0];

  float m_run = -INFINITY, l_run = 0.0f;
  float o_acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;

  int j = 0;
  bool timed_out = false;
  for (; j < n_mine; ++j) {
    const int s = j % STAGES;
    // table entry of the block this iteration will prefetch, loaded early
    const long long next_blk = (lane == 0 && j + STAGES < n_mine) ? phys(j + STAGES) : 0;
    if (!mbar_wait_bounded(&bar[s], (j / STAGES) & 1)) {
      timed_out = true;
      break;
    }
    const uint4* kb = reinterpret_cast<const uint4*>(ring + s * S::STAGE);
    const uint4* vb = reinterpret_cast<const uint4*>(ring + s * S::STAGE + kBlock * D);
    const int tok_base = (j_begin + warp + 4 * j) * kBlock;

    // keys: lane stream word nt*KS + ks holds channels 16ks + 4tig .. +3 of token 8nt + g
    uint32_t kw[2 * KS];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint4 x = kb[c * 32 + lane];
      kw[4 * c] = x.x;
      kw[4 * c + 1] = x.y;
      kw[4 * c + 2] = x.z;
      kw[4 * c + 3] = x.w;
    }
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.0f;
      if constexpr (QF) {
        // words (nt * (D/32) + kk) * 2 + {0, 1} are this lane's m16n8k32 B fragment
#pragma unroll
        for (int kk = 0; kk < QW; ++kk)
          mma_fp8_16832<FMT>(sacc[nt], qa[kk][0], 0u, qa[kk][1], 0u, kw[(nt * QW + kk) * 2],
                             kw[(nt * QW + kk) * 2 + 1]);
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t w = kw[nt * KS + ks];
          mma16816(sacc[nt], qa[ks][0], 0u, qa[ks][1], 0u, fp8_lo_pair<FMT>(w), fp8_hi_pair<FMT>(w));
        }
      }
    }
    float sc[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = tok_base + 8 * nt + 2 * tig + e;
        sc[2 * nt + e] = (tok < len) ? sacc[nt][e] * kmul : -INFINITY;
      }
    float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    mx = quad_max(mx);
    const float m_new = fmaxf(m_run, mx);
    if (m_new != m_run) {
      const float alpha = fast_exp2(m_run - m_new);
      l_run *= alpha;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o_acc[i][0] *= alpha;
        o_acc[i][1] *= alpha;
        o_acc[i][2] *= alpha;
        o_acc[i][3] *= alpha;
      }
      m_run = m_new;
    }
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = fast_exp2(sc[i] - m_new);
    l_run += (p[0] + p[1]) + (p[2] + p[3]);
    const __half2 h0 = __floats2half2_rn(p[0], p[1]), h1 = __floats2half2_rn(p[2], p[3]);
    const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
    const uint32_t A0 = h2_bits(h0), A1 = pack_rn_f16x2(p[0] - f0.x, p[1] - f0.y);
    const uint32_t A2 = h2_bits(h1), A3 = pack_rn_f16x2(p[2] - f1.x, p[3] - f1.y);

    // values: lane's stream word nt holds (r = 0, r = 1) byte pairs of channel 8nt + g
    uint32_t vw[NT];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint4 x = vb[c * 32 + lane];
      vw[4 * c] = x.x;
      vw[4 * c + 1] = x.y;
      vw[4 * c + 2] = x.z;
      vw[4 * c + 3] = x.w;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      mma16816(o_acc[nt], A0, A1, A2, A3, fp8_lo_pair<FMT>(vw[nt]), fp8_hi_pair<FMT>(vw[nt]));

    __syncwarp();
    if (lane == 0 && j + STAGES < n_mine) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(j + STAGES, next_blk);
    }
  }
  if (timed_out) {
    if (lane == 0) report_timeout(a.status);
    for (int jj = j; jj < n_mine && jj < j + STAGES; ++jj) (void)mbar_wait_bounded(&bar[jj % STAGES], (jj / STAGES) & 1);
    m_run = -INFINITY;
    l_run = 0.0f;
#pragma unroll
    for (int i = 0; i < NT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
  }
  l_run = quad_sum(l_run);

  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = 8 * nt + 2 * tig;
    o_s[(warp * 8 + g) * D + c] = (o_acc[nt][0] + o_acc[nt][2]) * vscale;
    o_s[(warp * 8 + g) * D + c + 1] = (o_acc[nt][1] + o_acc[nt][3]) * vscale;
  }
  if (tig == 0) {
    m_s[warp * 8 + g] = m_run;
    l_s[warp * 8 + g] = l_run;
  }
  __syncthreads();
  finish_split<D>(o_s, m_s, l_s, gq, static_cast<long long>(b) * a.q_heads + h * gq, split, a.splits, a.splits, a.part_o,
                  a.part_ml, a.counters + static_cast<long long>(b) * a.kv_heads + h, a.out, a.out_fp32);
}

constexpr int kFp8Stages = 4;

template <int D, int FMT, bool QF>
cudaError_t fp8_decode_dispatch(const Fp8DecodeArgs& a, cudaStream_t s) {
  constexpr int smem = Fp8Smem<D, kFp8Stages>::BYTES;
  auto kern = fp8_decode_kernel<D, kFp8Stages, FMT, QF>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.kv_heads, a.batch);
  kern<<<grid, 128, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
int fp8_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    constexpr int smem = Fp8Smem<D, kFp8Stages>::BYTES;
    auto kern = fp8_decode_kernel<D, kFp8Stages, 0, false>;  // every variant uses about the same resources
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, smem) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

int fp8_decode_blocks_per_sm(int head_dim) { return head_dim == 64 ? fp8_occupancy<64>() : fp8_occupancy<128>(); }

// Resident cast blocks per SM (the grid holds exactly that many: every warp
// then strides over the units with its copies one unit ahead).
int cast_blocks_per_sm(int head_dim) {
  static int cached[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 4;
  const int i = head_dim == 128 ? 1 : 0;
  if (cached[dev][i] == 0) {
    int n = 0;
    const cudaError_t e = head_dim == 128
                              ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp8_cast_kernel<128, 0>, 32 * kCastWarps, 0)
                              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp8_cast_kernel<64, 0>, 32 * kCastWarps, 0);
    cached[dev][i] = (e == cudaSuccess && n > 0) ? n : 4;
  }
  return cached[dev][i];
}

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, cudaStream_t s) {
  if (!a.static_scale) {
    const long long row_vecs = static_cast<long long>(a.seq_len) * a.head_dim / 8;
    const long long n_vec = static_cast<long long>(a.batch) * a.kv_heads * row_vecs;
    const int n_scales = a.per_head ? a.kv_heads : 1;
    fp8_amax_kernel<<<dim3(a.amax_blocks, n_scales), 256, 0, s>>>(reinterpret_cast<const uint4*>(a.x), n_vec,
                                                                   a.batch, a.kv_heads, row_vecs, a.amax_partials);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    fp8_scale_kernel<<<n_scales, 256, 0, s>>>(a.amax_partials, a.amax_blocks, a.fmt ? 57344.0f : 448.0f, a.scale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int nb = (a.seq_len + kBlock - 1) / kBlock;
  const long long units = static_cast<long long>(a.batch) * a.kv_heads * nb;
  const long long want = (units + kCastWarps - 1) / kCastWarps;
  const long long full = static_cast<long long>(cast_blocks_per_sm(a.head_dim)) * device_sm_count();
  const int grid = static_cast<int>(want < full ? want : full);
  switch (a.head_dim * 10 + a.fmt) {
    case 1280: fp8_cast_kernel<128, 0><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 1281: fp8_cast_kernel<128, 1><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 640: fp8_cast_kernel<64, 0><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 641: fp8_cast_kernel<64, 1><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_tensor_scale(const uint16_t* x, long long n_vec, float fmax, uint32_t* partials, int blocks,
                                float* scale, cudaStream_t s) {
  fp8_amax_kernel<<<dim3(blocks, 1), 256, 0, s>>>(reinterpret_cast<const uint4*>(x), n_vec, 1, 1, n_vec, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fp8_scale_kernel<<<1, 256, 0, s>>>(partials, blocks, fmax, scale);
  return cudaGetLastError();
}

cudaError_t launch_fp8_decode(const Fp8DecodeArgs& a, cudaStream_t s) {
  switch (a.head_dim * 100 + a.fmt * 10 + (a.q_fp8 ? 1 : 0)) {
    case 12800: return fp8_decode_dispatch<128, 0, false>(a, s);
    case 12810: return fp8_decode_dispatch<128, 1, false>(a, s);
    case 6400: return fp8_decode_dispatch<64, 0, false>(a, s);
    case 6410: return fp8_decode_dispatch<64, 1, false>(a, s);
    case 12801: return fp8_decode_dispatch<128, 0, true>(a, s);
    case 12811: return fp8_decode_dispatch<128, 1, true>(a, s);
    case 6401: return fp8_decode_dispatch<64, 0, true>(a, s);
    case 6411: return fp8_decode_dispatch<64, 1, true>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fp8_quantize_query(const Fp8QueryArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  const long long n_vec = a.n / 8;
  fp8_amax_kernel<<<dim3(a.amax_blocks, 1), 256, 0, s>>>(reinterpret_cast<const uint4*>(a.q), n_vec, 1, 1, n_vec,
                                                          a.partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long want = (n_vec + 255) / 256;
  const long long full = 2LL * device_sm_count();
  fp8_query_cast_kernel<<<static_cast<int>(want < full ? want : full), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
