// KIVI 2/4-bit KV cache kernels for sm_103a: group quantize + pack (prefill and
// residual flush) and token copies (window fill, append). The decode attention
// over the packed codes is in kivi_decode_tc.cu.
//
// Method: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 3
// (keys per channel, values per token, groups of 32 tokens, fp16 residual
// window flushed when full); affine form of "大模型量化从0到1（十三）：KV Cache 量化"
// (CSDN), section 10; attention softmax(q K^T / sqrt(d)) V of the same page,
// section 2, with grouped-query sharing (section 5).
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "kivi_layout.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// ---------------------------------------------------------------------------
// Group quantization (one thread block per (group, kv head, batch row))
// ---------------------------------------------------------------------------

// The group formula in IEEE fp32 with round-to-nearest-even everywhere.
__device__ __forceinline__ void group_scale_zero(float mn, float mx, float levels, __half& s16, __half& z16) {
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), levels));
  z16 = __float2half_rn(__fadd_rn(mn, 0.0f));  // exact; -0 becomes +0
}

// The group formula's code clamp(rint(fl32((x - z) / s)), 0, levels). The
// quotient comes from rcp = RN(1/s) and one correction step, bit-identical to
// the IEEE division here (x, z and s are fp16 values, so nothing under- or
// overflows; s = 0 has rcp = 0 and gives code 0 as the formula does), and
// rint + clamp are one round-to-nearest-even conversion (x >= z: no negative
// quotients) and a min.
__device__ __forceinline__ uint32_t group_code(float x, float zf, float sf, float rcp, uint32_t levels) {
  return min(__float2uint_rn(div_rn_by_rcp(__fsub_rn(x, zf), sf, rcp)), levels);
}

// One packed code word of a group (storage word u of lane (gg, tg)).
template <int D, int KB>
__device__ __forceinline__ uint32_t key_word(const __half* xk, int RS, const float* sk, const float* zk,
                                             const float* rk, int u, int gg, int tg) {
  constexpr uint32_t KL = (1u << KB) - 1u;
  uint32_t w = 0;
#pragma unroll
  for (int rr = 0; rr < (KB == 2 ? 2 : 1); ++rr) {
    const int ks = (KB == 2) ? u : (u >> 1);
    const int r = (KB == 2) ? rr : (u & 1);
    const int d0 = 16 * ks + 8 * r + 2 * tg;
    const float2 s01 = *reinterpret_cast<const float2*>(sk + d0), z01 = *reinterpret_cast<const float2*>(zk + d0),
                 r01 = *reinterpret_cast<const float2*>(rk + d0);
    const float s0 = s01.x, s1 = s01.y, z0 = z01.x, z1 = z01.y, r0 = r01.x, r1 = r01.y;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float2 x = __half22float2(reinterpret_cast<const __half2*>(xk)[(8 * nt + gg) * (RS / 2) + d0 / 2]);
      const int f = (KB == 2) ? ((4 * r + nt + 1) & 7) : nt;
      // fields never overlap: adding the shifted codes sets the same bits as or-ing them, and
      // w + (c << s) is one shift-and-add
      w += (group_code(x.x, z0, s0, r0, KL) << (KB * f)) + (group_code(x.y, z1, s1, r1, KL) << (16 + KB * f));
    }
  }
  return w;
}

// Value code word i of channel ch (the channel-major layout of include/kvq.h):
// field f of the word holds a pair of consecutive tokens, the first in the low
// half at bits [VB*f, VB*f + VB), the second in the high half. 4 bits: word i,
// field f = tokens 8i + 2f, +1. 2 bits: the decode exposes the fields of a word
// in the order (word, shift left 4, shift right 4, byte swap) at bits 6-7
// (tokens of the first 16, fields 3, 1, 5, 7) and 8-9 (tokens of the last 16,
// fields 4, 2, 6, 0), so field f holds tokens 16*kstep(f) + 8i + 2*idx(f), +1.
__device__ __forceinline__ int value_pair_token(int vb, int i, int f) {
  if (vb == 4) return 8 * i + 2 * f;
  const int kstep = (f & 1) ? 0 : 1;
  const int idx = (0x32200113 >> (4 * f)) & 0xF;  // f = 0..7 -> 3, 1, 1, 0, 0, 2, 2, 3
  return 16 * kstep + 8 * i + 2 * idx;
}

template <int D, int VB>
__device__ __forceinline__ uint32_t value_word(const __half* xv, int RS, const float* sv, const float* zv,
                                               const float* rv, int ch, int i) {
  constexpr uint32_t VL = (1u << VB) - 1u;
  uint32_t w = 0;
#pragma unroll
  for (int f = 0; f < 16 / VB; ++f) {
    const int t0 = value_pair_token(VB, i, f);
    const float x0 = __half2float(xv[t0 * RS + ch]), x1 = __half2float(xv[(t0 + 1) * RS + ch]);
    // fields never overlap: adding the shifted codes sets the same bits as or-ing them
    w += (group_code(x0, zv[t0], sv[t0], rv[t0], VL) << (VB * f)) +
         (group_code(x1, zv[t0 + 1], sv[t0 + 1], rv[t0 + 1], VL) << (16 + VB * f));
  }
  return w;
}

// Quantize and pack one group of 32 tokens of one (batch row, kv head): the
// fp16 rows k_src[0 .. 32*D) and v_src[...] (32 consecutive tokens of D
// channels) become the four records at kc, km, vc and vm. Run by a whole
// block of 128 threads.
template <int D, int KB, int VB>
__device__ __forceinline__ void quantize_group(const uint16_t* k_src, const uint16_t* v_src, uint8_t* kc, uint8_t* km,
                                               uint8_t* vc, uint8_t* vm) {
  using P = Kivi<D, KB, VB>;
  constexpr int RS = D + 8;  // padded row stride (halves): rows start 4 banks apart
  __shared__ __align__(16) __half xk[32 * RS];
  __shared__ __align__(16) __half xv[32 * RS];
  // scale, zero, RN(1/scale) per key channel and per value token (8-byte aligned: read in pairs)
  __shared__ __align__(8) float sk[D];
  __shared__ __align__(8) float zk[D];
  __shared__ __align__(8) float rk[D];
  __shared__ __align__(8) float sv[32];
  __shared__ __align__(8) float zv[32];
  __shared__ __align__(8) float rv[32];
  __shared__ uint16_t skb[D], zkb[D], svb[32], zvb[32];           // fp16 bits of scale and zero

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint4* srck = reinterpret_cast<const uint4*>(k_src);
  const uint4* srcv = reinterpret_cast<const uint4*>(v_src);
#pragma unroll
  for (int i = tid; i < 32 * D / 8; i += 128) {
    const int row = i / (D / 8), c8 = i % (D / 8);
    *reinterpret_cast<uint4*>(xk + row * RS + 8 * c8) = __ldcs(srck + i);
    *reinterpret_cast<uint4*>(xv + row * RS + 8 * c8) = __ldcs(srcv + i);
  }
  __syncthreads();

  constexpr float KL = static_cast<float>((1 << KB) - 1);
  constexpr float VL = static_cast<float>((1 << VB) - 1);

  if (tid < D / 2) {
    // keys: one pair of channels per thread, exact fp16 min/max over the 32 tokens
    const __half2* col = reinterpret_cast<const __half2*>(xk) + tid;
    __half2 mn = col[0], mx = col[0];
#pragma unroll 8
    for (int t = 1; t < 32; ++t) {
      const __half2 v = col[t * (RS / 2)];
      mn = __hmin2(mn, v);
      mx = __hmax2(mx, v);
    }
    const float2 mnf = __half22float2(mn), mxf = __half22float2(mx);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      __half s16, z16;
      group_scale_zero(e ? mnf.y : mnf.x, e ? mxf.y : mxf.x, KL, s16, z16);
      const int c = 2 * tid + e;
      sk[c] = __half2float(s16);
      zk[c] = __half2float(z16);
      rk[c] = (__half2float(s16) == 0.0f) ? 0.0f : __frcp_rn(__half2float(s16));
      skb[c] = __half_as_ushort(s16);
      zkb[c] = __half_as_ushort(z16);
    }
  } else if (warp >= 2) {
    // values: warps 2 and 3, two lanes per token, each over half of the row
    // with fp16 pair min/max; lane L reads its words in the order (c + L) mod
    // (D / 4), which keeps every shared-memory read conflict-free at D = 128
    constexpr int W2 = D / 4;                 // half2 words per lane
    const int t = 16 * (warp - 2) + (lane & 15), hh = lane >> 4;
    const __half2* row = reinterpret_cast<const __half2*>(xv) + t * (RS / 2) + hh * W2;
    __half2 mn = row[lane & (W2 - 1)], mx = mn;
#pragma unroll 8
    for (int c = 1; c < W2; ++c) {
      const __half2 v = row[(c + lane) & (W2 - 1)];
      mn = __hmin2(mn, v);
      mx = __hmax2(mx, v);
    }
    const float2 mnf2 = __half22float2(mn), mxf2 = __half22float2(mx);
    float mnf = fminf(mnf2.x, mnf2.y), mxf = fmaxf(mxf2.x, mxf2.y);
    mnf = fminf(mnf, __shfl_xor_sync(0xffffffffu, mnf, 16));
    mxf = fmaxf(mxf, __shfl_xor_sync(0xffffffffu, mxf, 16));
    if (hh == 0) {
      __half s16, z16;
      group_scale_zero(mnf, mxf, VL, s16, z16);
      sv[t] = __half2float(s16);
      zv[t] = __half2float(z16);
      rv[t] = (__half2float(s16) == 0.0f) ? 0.0f : __frcp_rn(__half2float(s16));
      svb[t] = __half_as_ushort(s16);
      zvb[t] = __half_as_ushort(z16);
    }
  }
  __syncthreads();

  // Code words, computed straight from the staged tile: warps 0-1 the key
  // words, warps 2-3 the value words. Key storage words 4*ug .. 4*ug + 3 of
  // fragment lane L are one 16-byte chunk (uint4 ug*32 + L); lane L of a warp
  // computes that chunk, so each shared-memory load of the warp has all 32
  // fragment lanes on the same word (conflict-free) and each store writes 512
  // contiguous bytes.
  if (warp < 2) {
    uint4* kdst = reinterpret_cast<uint4*>(kc);
    for (int ug = warp; ug < P::KW / 4; ug += 2) {
      uint4 w;
      w.x = key_word<D, KB>(xk, RS, sk, zk, rk, 4 * ug, lane >> 2, lane & 3);
      w.y = key_word<D, KB>(xk, RS, sk, zk, rk, 4 * ug + 1, lane >> 2, lane & 3);
      w.z = key_word<D, KB>(xk, RS, sk, zk, rk, 4 * ug + 2, lane >> 2, lane & 3);
      w.w = key_word<D, KB>(xk, RS, sk, zk, rk, 4 * ug + 3, lane >> 2, lane & 3);
      kdst[ug * 32 + lane] = w;
    }
  } else {
    // values, channel-major: thread c of warps 2-3 writes the VB words of channels c, c + 64, ...
    // (each shared-memory load of a warp reads 32 consecutive channels of one token row:
    // conflict-free; each store of a warp writes 32 * 4 * VB contiguous bytes)
    for (int ch = tid - 64; ch < D; ch += 64) {
      if constexpr (VB == 2) {
        uint2 w;
        w.x = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 0);
        w.y = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 1);
        reinterpret_cast<uint2*>(vc)[ch] = w;
      } else {
        uint4 w;
        w.x = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 0);
        w.y = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 1);
        w.z = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 2);
        w.w = value_word<D, VB>(xv, RS, sv, zv, rv, ch, 3);
        reinterpret_cast<uint4*>(vc)[ch] = w;
      }
    }
  }

  // Key meta: record ks*4 + tig = {s[d0], s[d0+1], s[d0+8], s[d0+9], z[...]}.
  if (tid < D / 4) {
    const int ks = tid >> 2, tg = tid & 3, d0 = 16 * ks + 2 * tg;
    uint4 rec;
    rec.x = skb[d0] | (static_cast<uint32_t>(skb[d0 + 1]) << 16);
    rec.y = skb[d0 + 8] | (static_cast<uint32_t>(skb[d0 + 9]) << 16);
    rec.z = zkb[d0] | (static_cast<uint32_t>(zkb[d0 + 1]) << 16);
    rec.w = zkb[d0 + 8] | (static_cast<uint32_t>(zkb[d0 + 9]) << 16);
    reinterpret_cast<uint4*>(km)[tid] = rec;
  } else if (tid >= 64 && tid < 72) {
    // Value meta: 4 records of scales, then 4 of zero points.
    const int i = tid - 64, tg = i & 3;
    const uint16_t* src = (i < 4) ? svb : zvb;
    uint4 rec;
    rec.x = src[2 * tg] | (static_cast<uint32_t>(src[2 * tg + 1]) << 16);
    rec.y = src[8 + 2 * tg] | (static_cast<uint32_t>(src[9 + 2 * tg]) << 16);
    rec.z = src[16 + 2 * tg] | (static_cast<uint32_t>(src[17 + 2 * tg]) << 16);
    rec.w = src[24 + 2 * tg] | (static_cast<uint32_t>(src[25 + 2 * tg]) << 16);
    reinterpret_cast<uint4*>(vm)[i] = rec;
  }
}

// Grid (groups, H_kv, B): group blockIdx.x of the source rows from src_tok0 on
// goes to group dst_group0 + blockIdx.x of the contiguous grouped region.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(128) kivi_quantize_kernel(QuantGroupsArgs a) {
  using P = Kivi<D, KB, VB>;
  const int grp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long long bh = static_cast<long long>(b) * a.kv_heads + h;
  const long long src_off = bh * a.src_bh_stride + static_cast<long long>(a.src_tok0 + 32 * grp) * D;
  const long long gi = bh * a.groups_cap + a.dst_group0 + grp;
  quantize_group<D, KB, VB>(a.k_src + src_off, a.v_src + src_off, a.k_codes + gi * P::KC, a.k_meta + gi * P::KM,
                            a.v_codes + gi * P::VC, a.v_meta + gi * P::VM);
}

// Grid (total groups, H_kv): item blockIdx.x is group x - begin[b] of sequence
// b's range, read from source token src0[b] + 32 * (x - begin[b]) and written
// to the pool block of logical group dst0[b] + (x - begin[b]), its four records
// back to back in the block's entry for kv head h. A block-table entry outside
// [0, num_blocks) is skipped: nothing is written for it.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(128) kivi_quantize_paged_kernel(PagedQuantArgs a) {
  using P = Kivi<D, KB, VB>;
  const int x = blockIdx.x, h = blockIdx.y;
  const int b = seq_of(a.r.begin, a.n_seqs, x);
  const int grp = x - a.r.begin[b];
  const long long bh = static_cast<long long>(b) * a.q.kv_heads + h;
  const long long src_off = bh * a.q.src_bh_stride + static_cast<long long>(a.r.src0[b] + 32 * grp) * D;
  const int blk = __ldg(a.pools.block_table + static_cast<long long>(b) * a.pools.groups_cap + a.r.dst0[b] + grp);
  if (blk < 0 || blk >= a.pools.num_blocks) return;
  uint8_t* e = a.q.k_codes + (static_cast<long long>(blk) * a.q.kv_heads + h) * P::STAGE;
  quantize_group<D, KB, VB>(a.q.k_src + src_off, a.q.v_src + src_off, e, e + P::KC, e + P::KC + P::KM,
                            e + P::KC + P::KM + P::VC);
}

// ---------------------------------------------------------------------------
// Token copies (fill the fp16 window, append a decode token, move a remainder)
// ---------------------------------------------------------------------------
__global__ void copy_tokens_kernel(CopyTokensArgs a) {
  // A decode launched right after this copy may start now: it reads what this
  // kernel writes (the fp16 window) only after its griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;");
  const int vec_per_tok = a.head_dim / 8;
  const long long per_bh = static_cast<long long>(a.n_tokens) * vec_per_tok;
  const long long total = per_bh * a.bh;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long bh = i / per_bh;
    const long long rem = i % per_bh;
    const long long tok = rem / vec_per_tok, v = rem % vec_per_tok;
    const long long s = (bh * a.src_bh_stride + (a.src_tok0 + tok) * a.head_dim) / 8 + v;
    const long long d = (bh * a.dst_bh_stride + (a.dst_tok0 + tok) * a.head_dim) / 8 + v;
    reinterpret_cast<uint4*>(a.k_dst)[d] = reinterpret_cast<const uint4*>(a.k_src)[s];
    reinterpret_cast<uint4*>(a.v_dst)[d] = reinterpret_cast<const uint4*>(a.v_src)[s];
  }
}

// Batched copies of a paged cache: token x of the launch (x < begin[n]) is
// token x - begin[b] of sequence b's range; for each kv head h its D channels
// go from source row src0[b] + (x - begin[b]) of (b, h) to window row
// dst0[b] + (x - begin[b]). Sources and destinations of one launch do not
// overlap.
__global__ void copy_tokens_paged_kernel(PagedCopyArgs a) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int vec_per_tok = a.c.head_dim / 8;
  const long long per_tok = static_cast<long long>(a.kv_heads) * vec_per_tok;
  const long long total = static_cast<long long>(a.r.begin[a.n_seqs]) * per_tok;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long x = i / per_tok, rem = i % per_tok;
    const int h = static_cast<int>(rem / vec_per_tok), v = static_cast<int>(rem % vec_per_tok);
    const int b = seq_of(a.r.begin, a.n_seqs, x);
    const long long tok = x - a.r.begin[b];
    const long long bh = static_cast<long long>(b) * a.kv_heads + h;
    const long long s = (bh * a.c.src_bh_stride + (a.r.src0[b] + tok) * a.c.head_dim) / 8 + v;
    const long long d = (bh * a.c.dst_bh_stride + (a.r.dst0[b] + tok) * a.c.head_dim) / 8 + v;
    reinterpret_cast<uint4*>(a.c.k_dst)[d] = reinterpret_cast<const uint4*>(a.c.k_src)[s];
    reinterpret_cast<uint4*>(a.c.v_dst)[d] = reinterpret_cast<const uint4*>(a.c.v_src)[s];
  }
}


template <int D, int KB, int VB>
cudaError_t quantize_dispatch(const QuantGroupsArgs& a, cudaStream_t s) {
  dim3 grid(a.n_groups, a.kv_heads, a.batch);
  kivi_quantize_kernel<D, KB, VB><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, int KB, int VB>
cudaError_t quantize_paged_dispatch(const PagedQuantArgs& a, cudaStream_t s) {
  dim3 grid(a.r.begin[a.n_seqs], a.q.kv_heads);
  kivi_quantize_paged_kernel<D, KB, VB><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kivi_quantize(const QuantGroupsArgs& a, cudaStream_t s) {
  if (a.n_groups <= 0) return cudaSuccess;
  const int key = a.head_dim * 100 + a.k_bits * 10 + a.v_bits;
  switch (key) {
    case 6422: return quantize_dispatch<64, 2, 2>(a, s);
    case 6424: return quantize_dispatch<64, 2, 4>(a, s);
    case 6442: return quantize_dispatch<64, 4, 2>(a, s);
    case 6444: return quantize_dispatch<64, 4, 4>(a, s);
    case 12822: return quantize_dispatch<128, 2, 2>(a, s);
    case 12824: return quantize_dispatch<128, 2, 4>(a, s);
    case 12842: return quantize_dispatch<128, 4, 2>(a, s);
    case 12844: return quantize_dispatch<128, 4, 4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_kivi_quantize_paged(const PagedQuantArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0 || a.r.begin[a.n_seqs] <= 0) return cudaSuccess;
  switch (a.q.head_dim * 100 + a.q.k_bits * 10 + a.q.v_bits) {
    case 6422: return quantize_paged_dispatch<64, 2, 2>(a, s);
    case 6424: return quantize_paged_dispatch<64, 2, 4>(a, s);
    case 6442: return quantize_paged_dispatch<64, 4, 2>(a, s);
    case 6444: return quantize_paged_dispatch<64, 4, 4>(a, s);
    case 12822: return quantize_paged_dispatch<128, 2, 2>(a, s);
    case 12824: return quantize_paged_dispatch<128, 2, 4>(a, s);
    case 12842: return quantize_paged_dispatch<128, 4, 2>(a, s);
    case 12844: return quantize_paged_dispatch<128, 4, 4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_copy_tokens_paged(const PagedCopyArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0 || a.r.begin[a.n_seqs] <= 0) return cudaSuccess;
  const long long total = static_cast<long long>(a.r.begin[a.n_seqs]) * a.kv_heads * (a.c.head_dim / 8);
  const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  copy_tokens_paged_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_copy_tokens(const CopyTokensArgs& a, cudaStream_t s) {
  if (a.n_tokens <= 0) return cudaSuccess;
  const long long total = static_cast<long long>(a.n_tokens) * (a.head_dim / 8) * a.bh;
  const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  copy_tokens_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace kvq
