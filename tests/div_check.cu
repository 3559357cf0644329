// The reciprocal-and-correction quotient used by the quantize kernels must be
// bit-identical to the IEEE division (__fdiv_rn) on the operands those kernels
// meet. Three sweeps, each counting mismatching quotients:
//   A: every positive finite fp16 scale s x every non-negative finite fp16 d;
//   B: d = x - z for random fp16 x >= z (an fp32 difference), random fp16 s,
//      and the half-integer quotients d = (k + 1/2) s and their neighbours;
//   C: every fp16 x (zeros, infinities and NaNs included) against random fp32
//      scales in [2^-96, 2^96], with the IEEE special values kept (the FP8
//      cast; any two NaNs count as equal: every NaN casts to the same byte).
// Built and run by tests/test_gpu_div.py.
#include <cstdio>
#include <cuda_fp16.h>

#include "kvq_device.cuh"

__device__ __forceinline__ unsigned long long mix(unsigned long long x) {  // splitmix64 finaliser
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

__device__ __forceinline__ bool same(float a, float b) { return __float_as_uint(a) == __float_as_uint(b); }

__device__ __forceinline__ float h2f(unsigned bits) { return __half2float(__ushort_as_half((unsigned short)bits)); }

// A: thread = one scale (fp16 bits 1 .. 0x7BFF), loop over every d in fp16 bits 0 .. 0x7BFF
__global__ void sweep_a(unsigned long long* bad) {
  const unsigned sb = 1 + blockIdx.x * blockDim.x + threadIdx.x;
  if (sb > 0x7BFFu) return;
  const float s = h2f(sb), y = __frcp_rn(s);
  unsigned long long n = 0;
  for (unsigned db = 0; db <= 0x7BFFu; ++db) {
    const float d = h2f(db);
    n += !same(kvq::div_rn_by_rcp(d, s, y), __fdiv_rn(d, s));
  }
  if (n) atomicAdd(bad, n);
}

// B: random fp32 differences and half-integer quotients
__global__ void sweep_b(unsigned long long* bad, unsigned long long per_thread) {
  const unsigned long long t = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
  unsigned long long n = 0;
  for (unsigned long long i = 0; i < per_thread; ++i) {
    const unsigned long long r = mix(t * per_thread + i);
    unsigned xb = r & 0x7FFFu, zb = (r >> 16) & 0x7FFFu, sb = 1 + ((r >> 32) % 0x7BFFu);
    if ((xb & 0x7C00u) == 0x7C00u) xb &= 0x7BFFu;  // keep x and z finite
    if ((zb & 0x7C00u) == 0x7C00u) zb &= 0x7BFFu;
    float x = h2f(xb | ((r >> 48) & 1u) << 15), z = h2f(zb | ((r >> 49) & 1u) << 15);
    if (x < z) { const float tmp = x; x = z; z = tmp; }
    const float s = h2f(sb), y = __frcp_rn(s);
    const float d = __fsub_rn(x, z);
    n += !same(kvq::div_rn_by_rcp(d, s, y), __fdiv_rn(d, s));
    // quotients at and beside k + 1/2 for the code levels
    const float k = (float)((r >> 50) & 15u) + 0.5f;
    const float dt = __fmul_rn(k, s);
    const float cand[3] = {dt, __uint_as_float(__float_as_uint(dt) + 1u), __uint_as_float(__float_as_uint(dt) - 1u)};
#pragma unroll
    for (int c = 0; c < 3; ++c) n += !same(kvq::div_rn_by_rcp(cand[c], s, y), __fdiv_rn(cand[c], s));
  }
  if (n) atomicAdd(bad, n);
}

// C: thread = one random scale, loop over every finite fp16 x
__global__ void sweep_c(unsigned long long* bad, int n_scales) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_scales) return;
  const unsigned long long r = mix(0xC0FFEEull + t);
  const int e = (int)(r % 193) - 96;                     // exponent in [-96, 96]
  const float s = ldexpf(1.0f + (float)((r >> 8) & 0x7FFFFF) * 0x1p-23f, e);
  const float y = __frcp_rn(s);
  unsigned long long n = 0;
  for (unsigned xb = 0; xb < 0x10000u; ++xb) {
    const float x = h2f(xb);
    const float got = kvq::div_rn_by_rcp_signed(x, s, y), want = __fdiv_rn(x, s);
    n += !(same(got, want) || (isnan(got) && isnan(want)));  // any NaN casts to the same byte
  }
  if (n) atomicAdd(bad, n);
}

int main() {
  unsigned long long* bad = nullptr;
  if (cudaMalloc(&bad, 3 * sizeof(unsigned long long)) != cudaSuccess) return 2;
  cudaMemset(bad, 0, 3 * sizeof(unsigned long long));
  sweep_a<<<(0x7BFF + 255) / 256, 256>>>(bad);
  const unsigned long long per_thread = 1024;
  sweep_b<<<1024, 256>>>(bad + 1, per_thread);
  const int n_scales = 8192;
  sweep_c<<<n_scales / 256, 256>>>(bad + 2, n_scales);
  cudaError_t err = cudaDeviceSynchronize();
  unsigned long long h[3] = {~0ull, ~0ull, ~0ull};
  cudaMemcpy(h, bad, sizeof(h), cudaMemcpyDeviceToHost);
  printf("A=%llu B=%llu C=%llu checked_A=%llu checked_B=%llu checked_C=%llu err=%s\n", h[0], h[1], h[2],
         (unsigned long long)0x7BFF * 0x7C00, 1024ull * 256 * per_thread * 4, (unsigned long long)n_scales * 65536,
         cudaGetErrorString(err));
  return 0;
}
