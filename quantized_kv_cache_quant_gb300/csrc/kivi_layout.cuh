// Record sizes of the packed KIVI cache and the bit fields its decode reads,
// shared by the quantize kernels (kivi_kernels.cu) and the decode kernel
// (kivi_decode_tc.cu). The byte layout itself is specified in include/kvq.h.
#pragma once

#include <cstdint>

namespace kvq {

template <int D, int KB, int VB>
struct Kivi {
  static constexpr int KS = D / 16;                      // k-steps of q . k^T
  static constexpr int KW = (KB == 2) ? D / 16 : D / 8;  // key code words per fragment lane
  static constexpr int VWC = VB;                         // value code words per channel (32 tokens)
  static constexpr int KC = 32 * D * KB / 8;             // bytes of one group's records
  static constexpr int KM = 4 * D;
  static constexpr int VC = 32 * D * VB / 8;
  static constexpr int VM = 128;
  static constexpr int STAGE = KC + KM + VC + VM;
  static_assert(STAGE % 16 == 0, "bulk copies need 16-byte multiples");
};

// Masks that keep the code field of each fp16 half after a shift: bits 6-7
// or 8-9 for 2-bit codes, bits 6-9 for 4-bit codes. The field then reads as
// the fp16 subnormal code * 2^(P-24), P = 6 or 8, which the tensor cores
// multiply exactly (the top mantissa bits keep full fp32-accumulation
// accuracy). A 2-bit word holds 8 fields per half; the word itself, its shifts
// by 4 either way and its per-half byte swap bring two fields each to bits 6-7
// and 8-9: three operations and eight masks for 16 codes.
constexpr uint32_t kMaskP6 = 0x00C000C0u;
constexpr uint32_t kMaskP8 = 0x03000300u;
constexpr uint32_t kMask4 = 0x03C003C0u;
constexpr float kInvP6 = 262144.0f;  // 2^18 = 2^(24-6)
constexpr float kInvP8 = 65536.0f;   // 2^16 = 2^(24-8)

// The sequence that owns item x of a batched launch: the b < n with
// begin[b] <= x < begin[b + 1] (begin is non-decreasing, begin[0] = 0 <= x <
// begin[n]). Binary search over the parameter array.
__device__ __forceinline__ int seq_of(const int* begin, int n, long long x) {
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

}  // namespace kvq
