// NVFP4 paged KV cache kernels for sm_103a: 4-bit E2M1 values with one E4M3
// scale per 16 channels of a token and one fp32 scale per tensor; cast +
// scatter into paged blocks, and split-K decode attention over the paged cache.
//
// Method: "大模型量化从0到1（十三）：KV Cache 量化" (CSDN), section 21.2 (NVFP4 KV
// cache: the more aggressive 4-bit floating-point path, scales calibrated
// offline, for Blackwell-class GPUs) and section 21.3 (about 1/4 of the BF16
// bytes); section 13 (paged blocks through a block table). The format is
// NVIDIA's public NVFP4; the tensor scale follows the pages' per-tensor rule
// scale = amax / FMAX with FMAX = 448 * 6 (the largest E4M3 block scale times
// the largest E2M1 value).
//   block scale byte b = E4M3(fl32(fl32(amax_b / 6) / s_t)),  S_b = e4m3(b)
//   code              = E2M1(fl32(x / fl32(S_b * s_t)))   (0 when S_b = 0)
//   dequantized value = e2m1(code) * S_b * s_t
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kBlock = 16;    // tokens per paged block
constexpr int kCastWarps = 4;

// Four fp32 pairs -> four bytes of E2M1 codes in one word (byte i from pair
// (lo[i], hi[i]), lo in the low nibble; round to nearest even, saturating).
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float2 (&q)[4]) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r)
      : "f"(q[0].x), "f"(q[0].y), "f"(q[1].x), "f"(q[1].y), "f"(q[2].x), "f"(q[2].y), "f"(q[3].x), "f"(q[3].y));
  return r;
}

// Byte k of w (two E2M1 codes, low nibble first) -> fp16x2 (exact).
template <int K>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
  uint32_t r;
  if constexpr (K == 0)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(r)
        : "r"(w));
  else if constexpr (K == 1)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
        : "=r"(r)
        : "r"(w));
  else if constexpr (K == 2)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
        : "=r"(r)
        : "r"(w));
  else
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
        : "=r"(r)
        : "r"(w));
  return r;
}

// The two E4M3 scale bytes of half h of w -> fp16x2 (exact).
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t w, int h) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(h ? (w >> 16) : (w & 0xFFFFu)));
}

// ---------------------------------------------------------------------------
// Cast + scatter: one warp per (b, h, logical block) unit, the units of a warp
// a grid-stride walk. Each warp stages the next unit's 16 x D fp16 values in
// its second shared-memory buffer with asynchronous copies (rows past the
// sequence zero-filled) while it casts the current one: the scale of each
// (token, 16-channel block), then the record, every lane its D/4 code bytes in
// 16-byte chunks (chunk c of lane l at byte (c*32 + l)*16), then the D scale
// bytes, in the in-block order of the role.
//
// Per element pair the quotient fl32(x / d), d = fl32(S_b * s_t), comes from
// y = RN(1/d) and one correction step in packed fp32 operations (exact for
// 2^-96 <= d <= 2^96; a unit with another nonzero d takes the IEEE division
// per element), and a block whose scale is 0 has its x masked to +0 first, so
// that all its codes are 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

// fl32(x / d) for each half of the fp16 pair xm (already masked), from the
// negated reciprocals ny = -RN(1/d): q0 = (-x)(-y) = fl32(x y), the residual
// r = fl32(d q0 - x) (the exact negation of the usual x - d q0, so the same
// value up to sign) and q = fl32(q0 - r y). Written with -x and -y the signed
// zeros come out right on their own: x = -0 gives -0, x = +0 gives +0.
__device__ __forceinline__ float2 quot_pair(uint32_t xm, float2 d, float2 ny) {
  const float2 nx = __half22float2(__hneg2(bits_h2(xm)));
  const float2 q0 = __fmul2_rn(nx, ny);
  const float2 r = __ffma2_rn(d, q0, nx);
  return __ffma2_rn(r, ny, q0);
}

template <int D, int ROLE>
__global__ void __launch_bounds__(32 * kCastWarps) nvfp4_cast_kernel(Nvfp4QuantArgs a) {
  constexpr int KS = D / 16;
  constexpr int RS = D + 8;  // padded row stride (halves): ldmatrix rows on distinct banks
  __shared__ __align__(16) __half tile[kCastWarps][2][kBlock * RS];
  // per (channel block, token) of the unit: d = fl32(S_b * s_t), ny = -RN(1/d) (-0 when d = 0) and
  // an fp16 mask (all ones when d > 0, else 0), in the order the role's element pairs read them:
  // keys {d, ny, mask, -} per token; values {d, d', ny, ny'} and {mask, mask'} per token pair
  constexpr int NPAR = (ROLE == 0) ? KS * kBlock : KS * kBlock / 2;
  __shared__ __align__(16) float4 par[kCastWarps][NPAR];
  __shared__ __align__(4) uint16_t msk[kCastWarps][KS * kBlock];  // values: [block][token]
  __shared__ uint8_t sbyte[kCastWarps][kBlock * KS];               // [token][block]: the E4M3 scale byte
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const float s_t = *a.scale;
  const bool st_fast = s_t >= 0x1p-96f && s_t <= 0x1p96f;
  const float y_t = st_fast ? __frcp_rn(s_t) : 0.0f;
  const float y_6 = __frcp_rn(6.0f);
  const int nb = (a.seq_len + kBlock - 1) / kBlock;
  const long long units = static_cast<long long>(a.batch) * a.kv_heads * nb;
  const long long stride = static_cast<long long>(gridDim.x) * kCastWarps;

  auto stage = [&](long long u, __half* xs) {
    const int j = static_cast<int>(u % nb);
    const long long bh = u / nb;
    const int t0 = j * kBlock, ntok = min(kBlock, a.seq_len - t0);
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (bh * a.seq_len + t0) * static_cast<long long>(D));
#pragma unroll
    for (int i = lane; i < kBlock * D / 8; i += 32) {
      const int tok = i / (D / 8), c8 = i % (D / 8);
      cp_async16_zfill(xs + tok * RS + 8 * c8, (tok < ntok) ? src + i : src, tok < ntok);
    }
  };

  long long u = blockIdx.x * static_cast<long long>(kCastWarps) + warp;
  if (u < units) stage(u, tile[warp][0]);
  cp_async_commit();
  for (int buf = 0; u < units; u += stride, buf ^= 1) {
    if (u + stride < units) stage(u + stride, tile[warp][buf ^ 1]);
    cp_async_commit();
    cp_async_wait_all_but_newest();
    __syncwarp();
    const __half* xs = tile[warp][buf];
    const int j = static_cast<int>(u % nb);
    const long long bh = u / nb;
    const int b = static_cast<int>(bh / a.kv_heads), h = static_cast<int>(bh % a.kv_heads);
    const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + j];
    if (blk >= 0 && blk < a.num_blocks) {  // uniform per warp: no write outside the pool
      // block scales
      bool slow = false, zero = false;  // a divisor outside the reciprocal range; a block whose scale is 0
#pragma unroll
      for (int p = lane; p < kBlock * KS; p += 32) {
        const int tok = p / KS, ks = p % KS;
        // the block's two 16-byte halves, the upper one first for odd ks / 4: the 8 lanes of a load
        // phase then cover all 32 banks (the blocks of a token are 32 bytes apart)
        const uint4* row = reinterpret_cast<const uint4*>(xs + tok * RS + 16 * ks);
        const int sw = (ks >> 2) & 1;
        const uint4 v0 = row[sw], v1 = row[sw ^ 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        // |x| as 15-bit patterns (ordered like the values), maxima of both halves at once
        uint32_t a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = w[k] & 0x7FFF7FFFu;
        const uint32_t m2 = __vimax3_u16x2(__vimax3_u16x2(a[0], a[1], a[2]), __vimax3_u16x2(a[3], a[4], a[5]),
                                           __vmaxu2(a[6], a[7]));
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        const float amax = __half2float(__ushort_as_half(static_cast<unsigned short>(m)));
        const float a6 = div_rn_by_rcp(amax, 6.0f, y_6);  // amax is a finite fp16 value: exact
        const float v = st_fast ? div_rn_by_rcp(a6, s_t, y_t) : __fdiv_rn(a6, s_t);
        const uint32_t byte = f32x2_to_e4m3x2(v, 0.0f) & 0xFFu;
        const float S = __half2float(__ushort_as_half(static_cast<unsigned short>(e4m3x2_to_f16x2(
            static_cast<uint16_t>(byte)) & 0xFFFFu)));
        const float d = __fmul_rn(S, s_t);
        const float ny = -((d > 0.0f) ? __frcp_rn(d) : 0.0f);
        sbyte[warp][p] = static_cast<uint8_t>(byte);
        if constexpr (ROLE == 0) {
          par[warp][ks * kBlock + tok] = make_float4(d, ny, __uint_as_float(d > 0.0f ? 0xFFFFFFFFu : 0u), 0.0f);
        } else {
          float* pv = reinterpret_cast<float*>(&par[warp][ks * (kBlock / 2) + (tok >> 1)]);
          pv[tok & 1] = d;
          pv[2 + (tok & 1)] = ny;
          msk[warp][ks * kBlock + tok] = (d > 0.0f) ? 0xFFFFu : 0u;
        }
        slow |= d > 0.0f && (d < 0x1p-96f || d > 0x1p96f);
        zero |= d == 0.0f;
      }
      slow = __any_sync(0xffffffffu, slow);
      zero = __any_sync(0xffffffffu, zero);
      __syncwarp();
      uint8_t* dst = a.pool + (static_cast<long long>(blk) * a.kv_heads + h) * (9 * D);
      const float4* pw = par[warp];
      const uint16_t* mw = msk[warp];
      // fl32(x / d) of one fp16 pair of elements: the reciprocal path, or (a unit with a block scale
      // outside its range) the IEEE division
      auto quot = [&](bool ieee, uint32_t xm, float2 d, float2 ny) -> float2 {
        if (!ieee) return quot_pair(xm, d, ny);
        const float2 x = __half22float2(bits_h2(xm));
        return make_float2(d.x == 0.0f ? 0.0f : __fdiv_rn(x.x, d.x), d.y == 0.0f ? 0.0f : __fdiv_rn(x.y, d.y));
      };
      // the lane's 16-byte chunks of codes; byte kk of chunk c = the codes of one fp16 pair of elements
      auto write_codes = [&](bool ieee, bool masked) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          float2 q[16];
          if constexpr (ROLE == 0) {
            // keys: byte p = (nt * KS + ks) * 2 + r holds channels 16 ks + 8 r + 2 tig, +1 of token 8 nt + g:
            // the (g, tig) element pair of the 8 x 8 tile of tokens 8 nt .., channels 8 (p % 2KS) .., four
            // tiles (consecutive p) per ldmatrix
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t t4[4];
              const int pl = 16 * c + 4 * q4 + (lane >> 3);  // the tile whose row this lane addresses
              ldsm_x4(t4, xs + (8 * (pl / (2 * KS)) + (lane & 7)) * RS + 8 * (pl % (2 * KS)));
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int kk = 4 * q4 + e, p = 16 * c + kk, nt = p / (2 * KS), ks = (p % (2 * KS)) >> 1;
                const float4 pr = pw[ks * kBlock + 8 * nt + g];
                q[kk] = quot(ieee, masked ? t4[e] & __float_as_uint(pr.z) : t4[e], make_float2(pr.x, pr.x),
                             make_float2(pr.y, pr.y));
              }
            }
          } else {
            // values: byte p = nt * 2 + r holds tokens 8 r + 2 tig, +1 of channel 8 nt + g, from the
            // transposed 8 x 8 tiles of tokens 8 r .., channels 8 nt .. (four tiles per ldmatrix)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int q4 = 0; q4 < 2; ++q4) {
                uint32_t t4[4];
                const int nt0 = 8 * c + 4 * q4;
                ldsm_x4_trans(t4, xs + (8 * r + (lane & 7)) * RS + 8 * (nt0 + (lane >> 3)));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int ta = 8 * r + 2 * tig, blkc = (8 * (nt0 + e) + g) >> 4;
                  const float4 pr = pw[blkc * (kBlock / 2) + (ta >> 1)];
                  const uint32_t xm = masked ? t4[e] & *reinterpret_cast<const uint32_t*>(mw + blkc * kBlock + ta) : t4[e];
                  q[(4 * q4 + e) * 2 + r] = quot(ieee, xm, make_float2(pr.x, pr.y), make_float2(pr.z, pr.w));
                }
              }
          }
          uint4 w;
          w.x = f32x8_to_e2m1x8({q[0], q[1], q[2], q[3]});
          w.y = f32x8_to_e2m1x8({q[4], q[5], q[6], q[7]});
          w.z = f32x8_to_e2m1x8({q[8], q[9], q[10], q[11]});
          w.w = f32x8_to_e2m1x8({q[12], q[13], q[14], q[15]});
          reinterpret_cast<uint4*>(dst)[c * 32 + lane] = w;
        }
      };
      // (warp-uniform) the usual unit: every divisor in the reciprocal range and none zero
      if (!slow && !zero)
        write_codes(false, false);
      else if (!slow)
        write_codes(false, true);
      else
        write_codes(true, true);
      // the D scale bytes: lane l writes bytes 4l .. 4l + 3 (D = 128) or 2l .. 2l + 1 (D = 64)
      constexpr int PER = D / 32;
      uint32_t sw = 0;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int s = PER * lane + e;  // scale byte index in the record
        int tok, blkc;
        if constexpr (ROLE == 0) {
          const int gg = s / (2 * KS), rem = s % (2 * KS), nt = rem / KS, ks = rem % KS;
          tok = 8 * nt + gg;
          blkc = ks;
        } else {
          const int ee = s & 1, jj = (s >> 1) % KS, tr = (s >> 1) / KS, r = tr & 1, tg = tr >> 1;
          tok = 8 * r + 2 * tg + ee;
          blkc = jj;
        }
        sw |= static_cast<uint32_t>(sbyte[warp][tok * KS + blkc]) << (8 * e);
      }
      if constexpr (PER == 4)
        reinterpret_cast<uint32_t*>(dst + 8 * D)[lane] = sw;
      else
        reinterpret_cast<uint16_t*>(dst + 8 * D)[lane] = static_cast<uint16_t>(sw);
    }
    __syncwarp();  // this buffer and the scale arrays are refilled by the next unit
  }
}

// ---------------------------------------------------------------------------
// Split-K decode attention over the paged NVFP4 cache. Grid (splits, H_kv, B),
// 4 warps; warp w of block x takes logical blocks x*bps + w, x*bps + w + 4,
// ... through a ring of STAGES stages (the key record and the value record of
// one kv head, 9*D bytes each) filled by bulk copies. Per m16n8k16 k-step the
// 16 key channels are one scale block, so every operand is fp16(e2m1 * S_b),
// exact (at most 6 significant bits, inside the fp16 range):
//   q.k^T : A = q (fp16), B = E2M1 keys converted to fp16, times the block
//           scale of their token (one half broadcast to both halves);
//           scores * s_t(K) * softmax scale.
//   p.V   : A = p split into fp16 hi + lo rows, B = E2M1 values as fp16 times
//           the scales of their two tokens (one E4M3 pair); outputs * s_t(V).
// kSwap (kv heads that serve at most 4 query heads): the operands change
// sides. The 16 tokens of a block (q.k^T) or 16 channels (p.V) are the tile
// rows and the query heads its 8 columns: column n of q.k^T carries head n/2
// (both columns of a head the same query, so lane (g, t) holds head t's scores
// of tokens g and g + 8), column n of p.V head n/2, part n%2 of p = hi + lo.
// The A fragments are the same record words the other arrangement reads as B
// fragments, regrouped (no layout change); half the MMAs and accumulators.
// ---------------------------------------------------------------------------
template <int D, int STAGES>
struct Nvfp4Smem {
  static constexpr int BAR_BYTES = 128;
  static constexpr int REC = 9 * D;
  static constexpr int STAGE = 2 * REC;
  static constexpr int RING = 4 * STAGES * STAGE;
  static constexpr int COMBINE = (4 * 8 * D + 64) * 4;
  static constexpr int AREA = RING > COMBINE ? RING : COMBINE;
  static constexpr int BYTES = BAR_BYTES + AREA;
};

// The reference max m_run moves only when a score exceeds it by more than this
// (log2 units), so the accumulators are rescaled rarely; the weights
// p <= 2^kNvfp4MaxSlack keep their fp16 hi + lo split exact to 2^-22 and the
// fp32 sums far from overflow.
constexpr float kNvfp4MaxSlack = 8.0f;
#ifndef KVQ_NVFP4_SWAP_MIN_BLOCKS
#define KVQ_NVFP4_SWAP_MIN_BLOCKS 4  // resident swapped-operand decode blocks per SM the registers are sized for
#endif

// Byte k (0..3, a compile-time value after unrolling) of w -> fp16x2.
__device__ __forceinline__ uint32_t e2m1_byte(uint32_t w, int k) {
  switch (k) {
    case 0: return e2m1x2_to_f16x2<0>(w);
    case 1: return e2m1x2_to_f16x2<1>(w);
    case 2: return e2m1x2_to_f16x2<2>(w);
    default: return e2m1x2_to_f16x2<3>(w);
  }
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t y) {
  return h2_bits(__hmul2(bits_h2(x), bits_h2(y)));
}

template <int D, int STAGES, bool kSwap>
__global__ void __launch_bounds__(128, kSwap ? KVQ_NVFP4_SWAP_MIN_BLOCKS : 1) nvfp4_decode_kernel(Nvfp4DecodeArgs a) {
  using S = Nvfp4Smem<D, STAGES>;
  constexpr int KS = D / 16, NT = D / 8, CH = D / 64;  // CH: 16-byte code chunks per lane
  constexpr int NACC = kSwap ? D / 16 : D / 8;         // p.V accumulator tiles
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
  // physical block of the warp's j-th logical block, clamped into the pool
  auto phys = [&](int j) -> long long {
    const int blk = table[j_begin + warp + 4 * j];
    return static_cast<long long>(min(max(blk, 0), a.num_blocks - 1));
  };
  auto issue = [&](int j, long long blk) {
    const long long off = (blk * a.kv_heads + h) * S::REC;
    uint8_t* dst = ring + (j % STAGES) * S::STAGE;
    uint64_t* bb = &bar[j % STAGES];
    mbar_arrive_expect_tx(bb, S::STAGE);
    bulk_g2s(dst, a.k_pool + off, S::REC, bb);
    bulk_g2s(dst + S::REC, a.v_pool + off, S::REC, bb);
  };
  if (lane == 0) {
    for (int j = 0; j < STAGES && j < n_mine; ++j) issue(j, phys(j));
  }

  // The query head of this lane's q fragments: row g (A), or column g (B, swapped).
  const int qh = kSwap ? (g >> 1) : g;
  const bool q_ok = qh < gq;
  const __half* qrow = reinterpret_cast<const __half*>(a.q) +
                       (static_cast<long long>(b) * a.q_heads + h * gq + (q_ok ? qh : 0)) * D;
  uint32_t qa[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
      qa[ks][jj] = q_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 * jj + 2 * tig) : 0u;
  const float kmul = *a.k_scale * a.scale_log2;
  const float vscale = *a.v_scale;

  float m_run = -INFINITY, l_run = 0.0f;
  float o_acc[NACC][4];
#pragma unroll
  for (int i = 0; i < NACC; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
  auto rescale = [&](float mx) {
    if (mx > m_run + kNvfp4MaxSlack) {
      const float alpha = fast_exp2(m_run - mx);
      l_run *= alpha;
#pragma unroll
      for (int i = 0; i < NACC; ++i) {
        o_acc[i][0] *= alpha;
        o_acc[i][1] *= alpha;
        o_acc[i][2] *= alpha;
        o_acc[i][3] *= alpha;
      }
      m_run = mx;
    }
  };

  int j = 0;
  bool timed_out = false;
  for (; j < n_mine; ++j) {
    const int s = j % STAGES;
    const long long next_blk = (lane == 0 && j + STAGES < n_mine) ? phys(j + STAGES) : 0;
    if (!mbar_wait_bounded(&bar[s], (j / STAGES) & 1)) {
      timed_out = true;
      break;
    }
    const uint8_t* kr = ring + s * S::STAGE;
    const uint8_t* vr = kr + S::REC;
    const int tok_base = (j_begin + warp + 4 * j) * kBlock;
    const bool ragged = tok_base + kBlock > len;  // the sequence's last block (warp-uniform)

    // keys: stream byte (nt*KS + ks)*2 + r holds channels 16ks + 8r + 2tig, +1 of
    // token 8nt + g; scale bytes nt*KS + ks of token 8nt + g, four to a word
    uint32_t kw[D / 16];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint4 x = reinterpret_cast<const uint4*>(kr)[c * 32 + lane];
      kw[4 * c] = x.x;
      kw[4 * c + 1] = x.y;
      kw[4 * c + 2] = x.z;
      kw[4 * c + 3] = x.w;
    }
    uint32_t ksw[KS / 2];
    if constexpr (D == 128) {
      const uint4 x = *reinterpret_cast<const uint4*>(kr + 8 * D + g * 2 * KS);
      ksw[0] = x.x;
      ksw[1] = x.y;
      ksw[2] = x.z;
      ksw[3] = x.w;
    } else {
      const uint2 x = *reinterpret_cast<const uint2*>(kr + 8 * D + g * 2 * KS);
      ksw[0] = x.x;
      ksw[1] = x.y;
    }
    // the fp16 codes of byte pair (i, r) times the scale of stream index i
    auto key_scale = [&](int i) {
      const uint32_t sp = e4m3_pair(ksw[i >> 2], (i >> 1) & 1);  // scales i & ~1, i | 1
      return h2_bits((i & 1) ? __high2half2(bits_h2(sp)) : __low2half2(bits_h2(sp)));
    };
    auto key_operand = [&](int i, int r) { return e2m1_byte(kw[i >> 1], 2 * (i & 1) + r); };

    // values: stream byte nt*2 + r holds tokens 8r + 2tig, +1 of channel 8nt + g;
    // scale pairs ((tig*2 + r)*KS + blk)*2 + {0, 1}, read as this lane's 4*KS bytes
    uint32_t vw[D / 16];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint4 x = reinterpret_cast<const uint4*>(vr)[c * 32 + lane];
      vw[4 * c] = x.x;
      vw[4 * c + 1] = x.y;
      vw[4 * c + 2] = x.z;
      vw[4 * c + 3] = x.w;
    }
    uint32_t vsw[KS];  // pair (r, blk) is half (r*KS + blk) of this array
    {
      const uint4* sp = reinterpret_cast<const uint4*>(vr + 8 * D + tig * 4 * KS);
#pragma unroll
      for (int c = 0; c < KS / 4; ++c) {
        const uint4 x = sp[c];
        vsw[4 * c] = x.x;
        vsw[4 * c + 1] = x.y;
        vsw[4 * c + 2] = x.z;
        vsw[4 * c + 3] = x.w;
      }
    }
    auto value_scale = [&](int r, int blk) {
      const int pr = r * KS + blk;
      return e4m3_pair(vsw[pr >> 1], pr & 1);
    };

    if constexpr (!kSwap) {
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int i = nt * KS + ks;
          const uint32_t sc2 = key_scale(i);
          mma16816(sacc[nt], qa[ks][0], 0u, qa[ks][1], 0u, hmul2_bits(key_operand(i, 0), sc2),
                   hmul2_bits(key_operand(i, 1), sc2));
        }
      }
      float sc[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) sc[2 * nt + e] = sacc[nt][e] * kmul;
      if (ragged) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (tok_base + 8 * (i >> 1) + 2 * tig + (i & 1) >= len) sc[i] = -INFINITY;
      }
      rescale(quad_max(fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]))));
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = fast_exp2(sc[i] - m_run);
      l_run += (p[0] + p[1]) + (p[2] + p[3]);
      const __half2 h0 = __floats2half2_rn(p[0], p[1]), h1 = __floats2half2_rn(p[2], p[3]);
      const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
      const uint32_t A0 = h2_bits(h0), A1 = pack_rn_f16x2(p[0] - f0.x, p[1] - f0.y);
      const uint32_t A2 = h2_bits(h1), A3 = pack_rn_f16x2(p[2] - f1.x, p[3] - f1.y);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t w = vw[nt >> 1];
        const uint32_t s0 = value_scale(0, nt >> 1), s1 = value_scale(1, nt >> 1);
        mma16816(o_acc[nt], A0, A1, A2, A3, hmul2_bits(e2m1_byte(w, 2 * (nt & 1)), s0),
                 hmul2_bits(e2m1_byte(w, 2 * (nt & 1) + 1), s1));
      }
    } else {
      // q.k^T: rows = tokens g, g + 8 (stream indices ks and KS + ks), k = channels of block ks
      float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t s_g = key_scale(ks), s_g8 = key_scale(KS + ks);
        mma16816(sacc, hmul2_bits(key_operand(ks, 0), s_g), hmul2_bits(key_operand(KS + ks, 0), s_g8),
                 hmul2_bits(key_operand(ks, 1), s_g), hmul2_bits(key_operand(KS + ks, 1), s_g8), qa[ks][0],
                 qa[ks][1]);
      }
      // head tig's scores of tokens g and g + 8 (columns 2tig + 1 repeat them)
      float sc0 = sacc[0] * kmul, sc1 = sacc[2] * kmul;
      if (ragged) {
        if (tok_base + g >= len) sc0 = -INFINITY;
        if (tok_base + 8 + g >= len) sc1 = -INFINITY;
      }
      rescale(col_max(fmaxf(sc0, sc1)));
      const float p0 = fast_exp2(sc0 - m_run), p1 = fast_exp2(sc1 - m_run);
      l_run += p0 + p1;
      // p = hi + lo in columns 2tig, 2tig + 1 of token rows g and g + 8, transposed
      // into the B fragments (k = tokens 2tig, +1 and 2tig + 8, +9; column g)
      const __half hi0 = __float2half_rn(p0), hi1 = __float2half_rn(p1);
      const __half lo0 = __float2half_rn(p0 - __half2float(hi0)), lo1 = __float2half_rn(p1 - __half2float(hi1));
      const uint32_t B0 = movm_trans(h2_bits(__halves2half2(hi0, lo0)));
      const uint32_t B1 = movm_trans(h2_bits(__halves2half2(hi1, lo1)));
      // p.V: rows = channels 16mt + g, + 8 (stream bytes 0, 2 / 1, 3 of word mt), k = tokens
#pragma unroll
      for (int mt = 0; mt < NACC; ++mt) {
        const uint32_t w = vw[mt];
        const uint32_t s0 = value_scale(0, mt), s1 = value_scale(1, mt);
        mma16816(o_acc[mt], hmul2_bits(e2m1_byte(w, 0), s0), hmul2_bits(e2m1_byte(w, 2), s0),
                 hmul2_bits(e2m1_byte(w, 1), s1), hmul2_bits(e2m1_byte(w, 3), s1), B0, B1);
      }
    }

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
    for (int i = 0; i < NACC; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
  }

  __syncthreads();
  if constexpr (!kSwap) {
    l_run = quad_sum(l_run);
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
  } else {
    // head tig: channels 16mt + g (columns hi, lo) and 16mt + 8 + g; rows gq.. of the warp's 8 are unused
    l_run = col_sum(l_run);
#pragma unroll
    for (int mt = 0; mt < NACC; ++mt) {
      o_s[(warp * 8 + tig) * D + 16 * mt + g] = (o_acc[mt][0] + o_acc[mt][1]) * vscale;
      o_s[(warp * 8 + tig) * D + 16 * mt + 8 + g] = (o_acc[mt][2] + o_acc[mt][3]) * vscale;
    }
    if (g == 0) {
      m_s[warp * 8 + tig] = m_run;
      l_s[warp * 8 + tig] = l_run;
    }
  }
  __syncthreads();
  finish_split<D>(o_s, m_s, l_s, gq, static_cast<long long>(b) * a.q_heads + h * gq, split, a.splits, a.splits, a.part_o,
                  a.part_ml, a.counters + static_cast<long long>(b) * a.kv_heads + h, a.out, a.out_fp32);
}

constexpr int kNvfp4Stages = 4;

// The swapped-operand arrangement serves kv heads with at most 4 query heads.
inline bool nvfp4_swapped(int gq) { return gq <= 4; }

template <int D, bool kSwap>
cudaError_t nvfp4_decode_dispatch(const Nvfp4DecodeArgs& a, cudaStream_t s) {
  constexpr int smem = Nvfp4Smem<D, kNvfp4Stages>::BYTES;
  auto kern = nvfp4_decode_kernel<D, kNvfp4Stages, kSwap>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.kv_heads, a.batch);
  kern<<<grid, 128, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool kSwap>
int nvfp4_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    constexpr int smem = Nvfp4Smem<D, kNvfp4Stages>::BYTES;
    auto kern = nvfp4_decode_kernel<D, kNvfp4Stages, kSwap>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, smem) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

int nvfp4_decode_blocks_per_sm(int head_dim, int gq) {
  if (nvfp4_swapped(gq)) return head_dim == 64 ? nvfp4_occupancy<64, true>() : nvfp4_occupancy<128, true>();
  return head_dim == 64 ? nvfp4_occupancy<64, false>() : nvfp4_occupancy<128, false>();
}

// Resident cast blocks per SM (occupancy API, once per device and variant).
int nvfp4_cast_blocks_per_sm(int head_dim, int role) {
  static int cached[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const int v = (head_dim == 128 ? 2 : 0) + (role ? 1 : 0);
  if (cached[dev][v] == 0) {
    int n = 0;
    cudaError_t e;
    switch (v) {
      case 3: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4_cast_kernel<128, 1>, 32 * kCastWarps, 0); break;
      case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4_cast_kernel<128, 0>, 32 * kCastWarps, 0); break;
      case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4_cast_kernel<64, 1>, 32 * kCastWarps, 0); break;
      default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4_cast_kernel<64, 0>, 32 * kCastWarps, 0); break;
    }
    cached[dev][v] = (e == cudaSuccess && n > 0) ? n : 1;
  }
  return cached[dev][v];
}

cudaError_t launch_nvfp4_quantize(const Nvfp4QuantArgs& a, cudaStream_t s) {
  if (!a.static_scale) {
    const long long n_vec = static_cast<long long>(a.batch) * a.kv_heads * a.seq_len * a.head_dim / 8;
    const cudaError_t e = launch_tensor_scale(a.x, n_vec, 448.0f * 6.0f, a.amax_partials, a.amax_blocks, a.scale, s);
    if (e != cudaSuccess) return e;
  }
  const int nb = (a.seq_len + kBlock - 1) / kBlock;
  const long long units = static_cast<long long>(a.batch) * a.kv_heads * nb;
  const long long want = (units + kCastWarps - 1) / kCastWarps;
  const long long full = static_cast<long long>(nvfp4_cast_blocks_per_sm(a.head_dim, a.role)) * device_sm_count();
  const int grid = static_cast<int>(want < full ? want : full);
  switch (a.head_dim * 10 + a.role) {
    case 1280: nvfp4_cast_kernel<128, 0><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 1281: nvfp4_cast_kernel<128, 1><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 640: nvfp4_cast_kernel<64, 0><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    case 641: nvfp4_cast_kernel<64, 1><<<grid, 32 * kCastWarps, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_decode(const Nvfp4DecodeArgs& a, cudaStream_t s) {
  if (a.kv_heads <= 0) return cudaErrorInvalidValue;
  const bool swapped = nvfp4_swapped(a.q_heads / a.kv_heads);
  switch (a.head_dim) {
    case 128: return swapped ? nvfp4_decode_dispatch<128, true>(a, s) : nvfp4_decode_dispatch<128, false>(a, s);
    case 64: return swapped ? nvfp4_decode_dispatch<64, true>(a, s) : nvfp4_decode_dispatch<64, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
