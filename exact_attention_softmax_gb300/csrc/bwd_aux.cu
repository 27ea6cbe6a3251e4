// bwd_aux.cu -- the bandwidth-bound steps around the backward main kernel:
//  * prep:    D_i = sum_c dO_ic * O_ic in fp32 for every query row (the row
//             statistic of the softmax Jacobian, dS = P * (dP - D)), and
//             optionally zero the fp32 dQ accumulator;
//  * convert: dQ = scale * dQ_acc rounded once to the input dtype.
// Rows are addressed through the same dense / packed rules as the forward,
// and D uses the LSE layout ([B,H,Lq] dense, [H,total] packed).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace sdpa {
namespace {

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Row r (0 <= r < rows) of the flattened query side -> (element offset, stat offset).
// Dense: r = (b*H + h)*Lq + i, element offset r*d, stat offset r.
// Packed: r = tok*H + h (memory order), stat offset h*total + tok.
__device__ __forceinline__ void row_offsets(const Problem& p, long long r, long long& elem, long long& stat) {
  elem = r * p.d;
  if (p.cu_seqlens == nullptr) {
    stat = r;
  } else {
    const long long tok = r / p.H, h = r % p.H;
    stat = h * p.Lq + tok;
  }
}

// One group of `lanes` threads per row, each lane covering 8 consecutive
// elements; the group reduces with shuffles.
template <typename T>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdProblem bp, long long rows, int lanes, int zero_acc) {
  const Problem& p = bp.f;
  const int rows_per_warp = 32 / lanes;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  const long long r = warp * rows_per_warp + lane / lanes;
  const int sub = lane % lanes;
  const bool live = r < rows;
  long long elem = 0, stat = 0;
  if (live) row_offsets(p, r, elem, stat);
  const T* O = static_cast<const T*>(p.o) + elem;
  const T* dO = static_cast<const T*>(bp.dO) + elem;
  float acc = 0.f;
  if (sizeof(T) == 2) {
    // fp16 / bf16 (d a multiple of 8, rows 16-byte aligned): one 16-byte load
    // of O and of dO per lane, and two 16-byte stores of zeros
    if (live && sub * 8 < p.d) {
      const uint4 ov = *reinterpret_cast<const uint4*>(O + sub * 8);
      const uint4 gv = *reinterpret_cast<const uint4*>(dO + sub * 8);
      const T* oe = reinterpret_cast<const T*>(&ov);
      const T* ge = reinterpret_cast<const T*>(&gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(to_f<T>(oe[e]), to_f<T>(ge[e]), acc);
      if (zero_acc) {
        float4* A = reinterpret_cast<float4*>(bp.dq_acc + elem + sub * 8);
        A[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        A[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else if (live) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = sub * 8 + e;
      if (c < p.d) acc = fmaf(to_f<T>(O[c]), to_f<T>(dO[c]), acc);
    }
    if (zero_acc) {
      float* A = bp.dq_acc + elem;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = sub * 8 + e;
        if (c < p.d) A[c] = 0.f;
      }
    }
  }
  for (int off = lanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0) bp.delta[stat] = acc;
}

// Eight elements per thread: two 16-byte loads, one 16-byte store (n is a
// multiple of 8 on the fp16 / bf16 path, whose head dims are 64 or 128).
template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, T* __restrict__ dq,
                                                         long long n, float scale) {
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (i + 7 < n) {
    const float4 a = *reinterpret_cast<const float4*>(acc + i);
    const float4 b = *reinterpret_cast<const float4*>(acc + i + 4);
    __align__(16) T out[8] = {from_f<T>(a.x * scale), from_f<T>(a.y * scale), from_f<T>(a.z * scale),
                              from_f<T>(a.w * scale), from_f<T>(b.x * scale), from_f<T>(b.y * scale),
                              from_f<T>(b.z * scale), from_f<T>(b.w * scale)};
    *reinterpret_cast<uint4*>(dq + i) = *reinterpret_cast<const uint4*>(out);
  } else {
    for (long long j = i; j < n; ++j) dq[j] = from_f<T>(acc[j] * scale);
  }
}

long long query_rows(const Problem& p) {
  return static_cast<long long>(p.cu_seqlens == nullptr ? p.B : 1) * p.H * p.Lq;
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdProblem& bp, int dtype, int zero_dq_acc, cudaStream_t s) {
  const Problem& p = bp.f;
  const long long rows = query_rows(p);
  if (rows == 0) return cudaSuccess;
  int lanes = 1;
  while (lanes * 8 < p.d) lanes *= 2;
  const long long threads = (rows + (32 / lanes) - 1) / (32 / lanes) * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (dtype == kF32) bwd_prep_kernel<float><<<blocks, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  else if (dtype == kF16) bwd_prep_kernel<__half><<<blocks, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  else bwd_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const BwdProblem& bp, int dtype, cudaStream_t s) {
  const Problem& p = bp.f;
  const long long n = query_rows(p) * p.d;
  if (n == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((n / 8 + 255) / 256 + 1);
  if (dtype == kF16)
    dq_convert_kernel<__half><<<blocks, 256, 0, s>>>(bp.dq_acc, static_cast<__half*>(bp.dq), n, p.scale);
  else
    dq_convert_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(bp.dq_acc, static_cast<__nv_bfloat16*>(bp.dq), n, p.scale);
  return cudaGetLastError();
}

}  // namespace sdpa
