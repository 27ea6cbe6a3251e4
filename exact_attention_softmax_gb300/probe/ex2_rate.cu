// ex2_rate.cu -- throughput probe of the exponential unit (not part of the
// attention library; the benchmark uses it to measure the ceiling that bounds
// the small-head-dim forward, which spends one ex2 per attention score).
//
// One CTA per SM, 16 warps (four per SM sub-partition), each thread running
// eight independent chains x <- 2^(-x), which converge to the fixed point
// near 0.64 and so stay finite for any number of steps. Each CTA reads the SM
// cycle counter after a block barrier at its start and end; the rate is the
// number of exponentials it computed over those cycles. Packed half-precision
// variants count two results per instruction.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr int kThreads = 512;
constexpr int kChains = 8;
constexpr int kMaxBlocks = 1024;

__device__ unsigned long long g_cycles[kMaxBlocks];
__device__ float g_sink[kMaxBlocks];

__device__ __forceinline__ float step_f32(float x) {
  float y;
  asm volatile("{\n\t.reg .f32 t;\n\tneg.f32 t, %1;\n\tex2.approx.ftz.f32 %0, t;\n\t}" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t step_f16x2(uint32_t x) {
  uint32_t y;
  asm volatile("{\n\t.reg .b32 t;\n\tneg.f16x2 t, %1;\n\tex2.approx.f16x2 %0, t;\n\t}" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t step_bf16x2(uint32_t x) {
  uint32_t y;
  asm volatile("{\n\t.reg .b32 t;\n\tneg.bf16x2 t, %1;\n\tex2.approx.ftz.bf16x2 %0, t;\n\t}" : "=r"(y) : "r"(x));
  return y;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) ex2_kernel(int iters) {
  float xf[kChains];
  uint32_t xh[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    xf[c] = 0.25f + 0.01f * c + 1e-4f * threadIdx.x;
    xh[c] = 0x34003400u + c;    // a pair of small positive halves
  }
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if (KIND == 0) xf[c] = step_f32(xf[c]);
      else if (KIND == 1) xh[c] = step_f16x2(xh[c]);
      else xh[c] = step_bf16x2(xh[c]);
    }
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += xf[c] + __uint_as_float(xh[c] & 0x3fffffffu);
  if (threadIdx.x == 0 && blockIdx.x < kMaxBlocks) {
    g_cycles[blockIdx.x] = t1 - t0;
    g_sink[blockIdx.x] = s;
  }
}

}  // namespace

// kind: 0 ex2.approx.ftz.f32, 1 ex2.approx.f16x2, 2 ex2.approx.ftz.bf16x2.
// Runs one CTA per SM (at most 1024 SMs) for `iters` steps of every chain on
// `stream` and synchronises it. Writes the exponentials per SM cycle of every
// CTA to per_sm[0 .. blocks) and the launch's device time (CUDA events) to
// *ms; returns the number of CTAs, or a negative value on a CUDA error.
extern "C" int sdpa_probe_ex2(int kind, int iters, double* per_sm, float* ms, void* stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (sms > kMaxBlocks) sms = kMaxBlocks;
  if (kind < 0 || kind > 2 || iters <= 0) return -2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t a, b;
  if (cudaEventCreate(&a) != cudaSuccess) return -1;
  if (cudaEventCreate(&b) != cudaSuccess) return -1;
  cudaEventRecord(a, s);
  if (kind == 0) ex2_kernel<0><<<sms, kThreads, 0, s>>>(iters);
  else if (kind == 1) ex2_kernel<1><<<sms, kThreads, 0, s>>>(iters);
  else ex2_kernel<2><<<sms, kThreads, 0, s>>>(iters);
  cudaEventRecord(b, s);
  if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(b) != cudaSuccess) return -1;
  cudaEventElapsedTime(ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  unsigned long long cyc[kMaxBlocks];
  if (cudaMemcpyFromSymbol(cyc, g_cycles, sizeof(unsigned long long) * sms) != cudaSuccess) return -1;
  const double per_block = static_cast<double>(kThreads) * kChains * iters * (kind == 0 ? 1 : 2);
  for (int i = 0; i < sms; ++i) per_sm[i] = cyc[i] ? per_block / static_cast<double>(cyc[i]) : 0.0;
  return sms;
}
