// Device-side building blocks shared by the kernels of libkvq: inline PTX for
// mbarriers, bulk (TMA) copies, the m16n8k16 tensor-core MMA and fp8
// conversions, plus a bounded wait that reports a timeout instead of hanging.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace kvq {

constexpr int kGroup = 32;               // tokens per KIVI group
constexpr uint32_t kStatusTimeout = 1u;  // status bit: a device wait gave up
constexpr int kWsHeader = 256;           // bytes reserved at the start of a decode workspace
constexpr int kMaxSplits = 64;           // split-K partials per (batch row, query head)
constexpr int kMaxGqa = 8;               // query heads per kv head handled by one MMA tile
constexpr int kChunkUnits = 6;           // decode work units (groups) one 32-token window chunk is charged
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait
// The decode splits each p * s_t (and each softmax weight p of a window
// token) into fp16 hi + lo tensor-core operands on separate accumulator rows
// or columns. The lo part is carried times kLoGain and its accumulator scaled
// back once at the end: a product below fp16's normal range (a token whose
// value scale is an fp16 subnormal) then keeps 11 more bits than the
// subnormal grid 2^-24 gives. |lo| <= half an ulp of hi <= 16, so
// |lo| * kLoGain <= 2^15 stays finite.
constexpr float kLoGain = 2048.0f;
constexpr float kLoGainInv = 1.0f / 2048.0f;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`; gives up after kWaitLimitNs and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// One bulk copy global -> shared (the 1-D form of the tensor memory accelerator);
// completion is counted in bytes on `bar`. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators.
// A (row-major 16x16): a0 = (row g, cols 2t,2t+1), a1 = (row g+8, same cols),
//                      a2 = (row g, cols 2t+8, 2t+9), a3 = (row g+8, cols 2t+8, 2t+9)
// B (16x8, "col"):     b0 = (rows 2t, 2t+1 of col g), b1 = (rows 2t+8, 2t+9 of col g)
// C/D:                 c0, c1 = (row g, cols 2t, 2t+1), c2, c3 = (row g+8, cols 2t, 2t+1)
// with g = lane / 4 and t = lane % 4.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 fp16 tiles from shared memory into mma.sync operand registers.
// Lane l gives the address of row l % 8 of tile l / 8 (16 contiguous bytes);
// register i then holds tile i in fragment order: lane (g, t) receives row g,
// columns 2t and 2t+1 (ldsm_x4), or with the tile transposed, rows 2t and
// 2t+1 of column g (ldsm_x4_trans).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* row) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* row) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a)
               : "memory");
}

// 16-byte asynchronous global -> shared copies (L2 only), committed in groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most one group (the newest) of this thread's copies is in flight
__device__ __forceinline__ void cp_async_wait_all_but_newest() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// The correctly rounded fp32 quotient d / s from y = RN(1/s), by Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; Handbook of
// Floating-Point Arithmetic, the chapter on division with an FMA): q0 =
// RN(d * y) is within an ulp of d / s, the residual r = d - s * q0 is exact
// with an FMA, and RN(q0 + r * y) = RN(d / s) as long as d, s and the quotient
// are normal or zero (no underflow or overflow). s = 0 with y = 0 gives 0. A
// zero numerator gives +0: the IEEE quotient of -0 is -0, so a caller that
// keeps the sign of zero restores it (div_rn_by_rcp_signed).
__device__ __forceinline__ float div_rn_by_rcp(float d, float s, float y) {
  const float q0 = __fmul_rn(d, y);
  const float r = __fmaf_rn(-q0, s, d);
  return __fmaf_rn(r, y, q0);
}
// The same for s > 0 with the IEEE results at the numerator's special values:
// the sign of a zero numerator kept (for s > 0 the quotient has the
// numerator's sign, so the copy changes nothing else) and an infinite
// numerator returned as is (the correction step would turn it into a NaN).
__device__ __forceinline__ float div_rn_by_rcp_signed(float d, float s, float y) {
  return isinf(d) ? d : copysignf(div_rn_by_rcp(d, s, y), d);
}

// c + a.lo * b.lo + a.hi * b.hi with fp16 halves and an fp32 accumulator
// (the fp16 products are exact in fp32; each add rounds once).
__device__ __forceinline__ float dot2_f16_f32(uint32_t a, uint32_t b, float c) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two fp32 values -> fp16x2 bits (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_rn_f16x2(float lo, float hi) {
  return h2_bits(__floats2half2_rn(lo, hi));
}

// Two E4M3 bytes (low byte first) -> fp16x2 bits (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Two fp32 values -> two E4M3 bytes (round to nearest even, saturating to
// +-448, NaN -> 0x7F); `lo` goes to the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E5M2 bytes (low byte first) -> fp16x2 bits. E5M2 has fp16's sign and
// exponent fields and the top two of its mantissa bits, so each byte becomes
// the high byte of its half (exact for every code, subnormals, infinities and
// NaNs included): one byte permute, bytes (0, b0, 0, b1).
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint16_t v) {
  return __byte_perm(static_cast<uint32_t>(v), 0u, 0x1404u);
}

// Two fp32 values -> two E5M2 bytes (round to nearest even, saturating to
// +-57344, NaN -> 0x7F); `lo` goes to the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// FP8 format FMT: 0 = E4M3, 1 = E5M2.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint16_t v) {
  if constexpr (FMT == 0)
    return e4m3x2_to_f16x2(v);
  else
    return e5m2x2_to_f16x2(v);
}
template <int FMT>
__device__ __forceinline__ uint16_t f32x2_to_fp8x2(float lo, float hi) {
  if constexpr (FMT == 0)
    return f32x2_to_e4m3x2(lo, hi);
  else
    return f32x2_to_e5m2x2(lo, hi);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Max and sum over the eight lanes that share t = lane % 4 (one column of an
// mma fragment: in the swapped-operand decodes, one query head's tokens).
__device__ __forceinline__ float col_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float col_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// Transpose of an 8 x 8 fp16 tile held in mma fragment order across the warp:
// lane (g, t) holds row g, columns 2t and 2t + 1 before and after.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void report_timeout(uint32_t* status) {
  if (status != nullptr) atomicOr(status, kStatusTimeout);
}

}  // namespace kvq

namespace kvq {

// Epilogue shared by the split-K decode kernels. The four warps of a thread
// block have left per-warp (m, l, o) in shared memory (o_s[4][8][D],
// m_s[4][8], l_s[4][8], log2 units). The block combines them and writes its
// partial `split` of each query row (slot row * stride + split); the last of
// the `splits_total` blocks of a (batch row, kv head) to finish — found with an
// atomic counter, no waiting — merges all splits into `out` and resets the
// counter for the next call.
// Needs blockDim.x == 128 and D in {64, 128}.
template <int D>
__device__ __forceinline__ void finish_split(float* o_s, float* m_s, float* l_s, int gq, long long q_row0, int split,
                                             int splits_total, int stride, float* part_o, float* part_ml,
                                             uint32_t* counter, void* out, int out_fp32) {
  const int tid = threadIdx.x;
  for (int i = tid; i < gq * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * 8 + r]);
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = fast_exp2(m_s[w * 8 + r] - M);
        L = fmaf(l_s[w * 8 + r], f, L);
        O = fmaf(o_s[(w * 8 + r) * D + c], f, O);
      }
    }
    const long long row = (q_row0 + r) * stride + split;
    part_o[row * D + c] = O;
    if (c == 0) {
      part_ml[row * 2] = M;
      part_ml[row * 2 + 1] = L;
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (tid == 0) last = (atomicAdd(counter, 1u) == static_cast<uint32_t>(splits_total - 1));
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) *counter = 0u;
  // merge weights per query row into shared memory (o_s is free now); one
  // warp per row, each lane holds splits lane and lane + 32 (kMaxSplits = 64)
  static_assert(kMaxSplits <= 64, "two splits per lane");
  float* wgt = o_s;                      // [8][kMaxSplits]
  float* inv_l = o_s + 8 * kMaxSplits;   // [8]
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < gq; r += blockDim.x >> 5) {
    const long long base = (q_row0 + r) * stride;
    float mv[2], lv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int sp = lane + 32 * k;
      mv[k] = (sp < splits_total) ? __ldcg(part_ml + (base + sp) * 2) : -INFINITY;
      lv[k] = (sp < splits_total) ? __ldcg(part_ml + (base + sp) * 2 + 1) : 0.0f;
    }
    const float M = warp_max(fmaxf(mv[0], mv[1]));
    float L = 0.0f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int sp = lane + 32 * k;
      const float f = (M == -INFINITY || sp >= splits_total) ? 0.0f : fast_exp2(mv[k] - M);
      if (sp < splits_total) wgt[r * kMaxSplits + sp] = f;
      L = fmaf(f, lv[k], L);
    }
    L = warp_sum(L);
    if (lane == 0) inv_l[r] = (L > 0.0f) ? 1.0f / L : 0.0f;
  }
  __syncthreads();
  // thread t sums column t % D of rows t / D, t / D + 128 / D, ...: the loads of
  // all its rows for one split are independent and are in flight together
  constexpr int kRowStep = 128 / D;
  constexpr int kRowsPer = (kMaxGqa + kRowStep - 1) / kRowStep;
  const int c = tid % D, r0 = tid / D;
  float O[kRowsPer];
#pragma unroll
  for (int k = 0; k < kRowsPer; ++k) O[k] = 0.0f;
#pragma unroll 4
  for (int sp = 0; sp < splits_total; ++sp) {
#pragma unroll
    for (int k = 0; k < kRowsPer; ++k) {
      const int r = r0 + k * kRowStep;
      if (r < gq) O[k] = fmaf(wgt[r * kMaxSplits + sp], __ldcg(part_o + ((q_row0 + r) * stride + sp) * D + c), O[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < kRowsPer; ++k) {
    const int r = r0 + k * kRowStep;
    if (r >= gq) continue;
    const long long o_idx = (q_row0 + r) * D + c;
    const float v = O[k] * inv_l[r];
    if (out_fp32)
      reinterpret_cast<float*>(out)[o_idx] = v;
    else
      reinterpret_cast<__half*>(out)[o_idx] = __float2half_rn(v);
  }
}

}  // namespace kvq
