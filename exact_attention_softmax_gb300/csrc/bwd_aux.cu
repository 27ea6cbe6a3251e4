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

// Row offsets. Dense: unit u = b*H + h holds rows r = u*Lq + i of the
// contiguous fp32 dQ accumulator (offset r*d) and of the statistics (offset
// r); its tensors are addressed at their strides. Packed: r = tok*H + h
// (memory order, every tensor [total, H, d]), statistic at h*total + tok.
__device__ __forceinline__ long long packed_stat(const Problem& p, long long r) {
  const long long tok = r / p.H, h = r % p.H;
  return h * p.Lq + tok;
}

// One group of `lanes` threads per row, each lane covering 8 consecutive
// elements; the group reduces with shuffles. Dense: blockIdx.y walks the
// (batch, head) units and x the rows of a unit, so no thread divides by a
// run-time size; packed: x walks all rows.
template <typename T>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdProblem bp, long long rows_per_unit, int lanes, int zero_acc) {
  const Problem& p = bp.f;
  const bool dense = p.cu_seqlens == nullptr;
  const int units = dense ? p.B * p.H : 1;
  const int rows_per_warp = 32 / lanes;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  const long long i = warp * rows_per_warp + lane / lanes;    // row within the unit
  const int sub = lane % lanes;
  for (int u = blockIdx.y; u < units; u += gridDim.y) {
    const bool live = i < rows_per_unit;
    const long long r = static_cast<long long>(u) * rows_per_unit + i;
    long long eo = 0, edo = 0;
    if (live) {
      eo = p.strided ? dense_off(p, kTo, u / p.H, u % p.H, i) : r * p.d;
      edo = p.strided ? dense_off(p, kTdo, u / p.H, u % p.H, i) : r * p.d;
    }
    const long long elem = r * p.d;
    const T* O = static_cast<const T*>(p.o) + eo;
    const T* dO = static_cast<const T*>(bp.dO) + edo;
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
        if (zero_acc && SDPA_CHECK(elem + sub * 8 + 8 <= bp.acc_rows * p.d, p.status)) {
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
      if (zero_acc && SDPA_CHECK(elem + p.d <= bp.acc_rows * p.d, p.status)) {
        float* A = bp.dq_acc + elem;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = sub * 8 + e;
          if (c < p.d) A[c] = 0.f;
        }
      }
    }
    for (int off = lanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const long long di = dense ? r : packed_stat(p, r);
    if (live && sub == 0 && SDPA_CHECK(di < bp.acc_rows, p.status)) bp.delta[di] = acc;
  }
}

// Eight elements of one row per thread (the fp16 / bf16 head dims, 32, 64
// or 128, are multiples of 8): two 16-byte loads of the contiguous accumulator,
// one 16-byte store into dQ at its strides. Dense: blockIdx.y walks the units
// and x the chunks of a unit; packed ([total, H, d], contiguous): x walks all.
template <typename T, int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BwdProblem bp, long long chunks_per_unit) {
  const Problem& p = bp.f;
  const bool dense = p.cu_seqlens == nullptr;
  const int units = dense ? p.B * p.H : 1;
  constexpr int kChunks = D / 8;                           // chunks per row
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= chunks_per_unit) return;
  const long long i = t / kChunks;                         // row within the unit
  const int c = static_cast<int>(t % kChunks) * 8;
  const float scale = p.scale;
  for (int u = blockIdx.y; u < units; u += gridDim.y) {
    const long long a_off = (static_cast<long long>(u) * chunks_per_unit + t) * 8;
    const long long q_off = p.strided ? dense_off(p, kTdq, u / p.H, u % p.H, i) + c : a_off;
    if (!SDPA_CHECK(a_off + 8 <= bp.acc_rows * D && q_off + 8 <= p.ext[kTdq], p.status)) continue;
    const float4 a = *reinterpret_cast<const float4*>(bp.dq_acc + a_off);
    const float4 b = *reinterpret_cast<const float4*>(bp.dq_acc + a_off + 4);
    __align__(16) T out[8] = {from_f<T>(a.x * scale), from_f<T>(a.y * scale), from_f<T>(a.z * scale),
                              from_f<T>(a.w * scale), from_f<T>(b.x * scale), from_f<T>(b.y * scale),
                              from_f<T>(b.z * scale), from_f<T>(b.w * scale)};
    *reinterpret_cast<uint4*>(static_cast<T*>(bp.dq) + q_off) = *reinterpret_cast<const uint4*>(out);
  }
}

// Rows of one unit (dense) or of the whole packed batch.
long long rows_per_unit(const Problem& p) {
  return p.cu_seqlens == nullptr ? static_cast<long long>(p.Lq) : static_cast<long long>(p.H) * p.Lq;
}

unsigned unit_blocks(const Problem& p) {
  const long long u = p.cu_seqlens == nullptr ? static_cast<long long>(p.B) * p.H : 1;
  return static_cast<unsigned>(u < 65535 ? u : 65535);
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdProblem& bp, int dtype, int zero_dq_acc, cudaStream_t s) {
  const Problem& p = bp.f;
  const long long rows = rows_per_unit(p);
  if (rows == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  int lanes = 1;
  while (lanes * 8 < p.d) lanes *= 2;
  const long long threads = (rows + (32 / lanes) - 1) / (32 / lanes) * 32;
  const dim3 grid(static_cast<unsigned>((threads + 255) / 256), unit_blocks(p));
  if (dtype == kF32) bwd_prep_kernel<float><<<grid, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  else if (dtype == kF16) bwd_prep_kernel<__half><<<grid, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  else bwd_prep_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(bp, rows, lanes, zero_dq_acc);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const BwdProblem& bp, int dtype, cudaStream_t s) {
  const Problem& p = bp.f;
  const long long chunks = rows_per_unit(p) * p.d / 8;
  if (chunks == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((chunks + 255) / 256), unit_blocks(p));
  if (p.d == 32) {
    if (dtype == kF16) dq_convert_kernel<__half, 32><<<grid, 256, 0, s>>>(bp, chunks);
    else dq_convert_kernel<__nv_bfloat16, 32><<<grid, 256, 0, s>>>(bp, chunks);
  } else if (p.d == 64) {
    if (dtype == kF16) dq_convert_kernel<__half, 64><<<grid, 256, 0, s>>>(bp, chunks);
    else dq_convert_kernel<__nv_bfloat16, 64><<<grid, 256, 0, s>>>(bp, chunks);
  } else if (p.d == 128) {
    if (dtype == kF16) dq_convert_kernel<__half, 128><<<grid, 256, 0, s>>>(bp, chunks);
    else dq_convert_kernel<__nv_bfloat16, 128><<<grid, 256, 0, s>>>(bp, chunks);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace sdpa
