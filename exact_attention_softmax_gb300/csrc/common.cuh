// common.cuh -- definitions shared by the C-ABI layer and the kernels of the
// GB300 exact-attention library (internal; not part of the public header).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa {

constexpr unsigned kStatusTimeout = 1u;  // == SDPA_STATUS_TIMEOUT
constexpr unsigned kStatusSeqlen = 2u;   // == SDPA_STATUS_SEQLEN
constexpr unsigned kStatusBounds = 4u;   // == SDPA_STATUS_BOUNDS (debug build only)
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per mbarrier wait

// Debug switches (testing only; zero in normal use).
constexpr int kDebugDropQArrive = 1;  // forward producer never loads Q: every wait times out
constexpr int kDebugShortO = 2;       // debug build: O's extent one row short, so the
                                      // last row's bounds check fails (its store is skipped)

// Debug build (-DSDPA_DEBUG): device-side bounds checks on the kernels'
// stores, reductions and shared-memory staging. A failed check sets
// kStatusBounds in the status word and the guarded access is skipped: nothing
// traps, and the host reports the bit. In the normal build a check is the
// constant true and costs nothing.
#ifdef SDPA_DEBUG
#define SDPA_CHECK(cond, status) (::sdpa::bounds_ok((cond), (status)))
#else
#define SDPA_CHECK(cond, status) true
#endif

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// Tensors of a call, for their dense-layout strides (Problem::st).
enum Tensor : int { kTq = 0, kTk, kTv, kTo, kTdo, kTdq, kTdk, kTdv, kTensors };

// One attention problem as the kernels see it. Dense: q/o [B,H,Lq,d],
// k/v [B,H,Lk,d] at any element strides (Problem::st), lse [B,H,Lq]. Packed (cu_seqlens != nullptr): B sequences;
// q/o [Lq = total query tokens, H, d] with sequence s at rows
// cu_seqlens[s]..cu_seqlens[s+1]; k/v [total_k, H, d] with rows from cu_k
// (cu_k == cu_seqlens for self-attention); lse [H, Lq]; max_q and Lk bound the
// query and key lengths of every sequence.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Lq, Lk, d;
  float scale;
  int causal;
  const int* cu_seqlens;
  const int* cu_k;
  int total_k;
  int max_q;
  unsigned* status;  // device status word (bit flags above)
  int debug;
  // Block-sparse attention (dense layout only): 0/1 per (128-query block,
  // 128-key block) at bmask[b * bm_sb + h * bm_sh + qb * bm_sq + kb], or NULL.
  const unsigned char* bmask;
  long long bm_sb, bm_sh;
  int bm_sq;
  // Additive mask (dense layout only): element (b, h, i, j) at
  // amask[b * am_sb + h * am_sh + i * am_sq + j], in the input dtype, or NULL.
  const void* amask;
  long long am_sb, am_sh, am_sq;
  // Dropout (dense layout only): score (i, j) of unit u is kept iff byte
  // j % 16 of Philox4x32-10(counter (j / 16, i, u, 0), key (seed_lo, seed_hi))
  // is at least drop_t; kept probabilities are scaled by drop_scale.
  int dropout;                 // 0 / 1
  unsigned drop_t;             // round(p * 256), 0..255
  float drop_scale;            // 256 / (256 - drop_t)
  unsigned seed_lo, seed_hi;
  // Dense layout: element strides (batch, head, row) of every tensor of the
  // call, indexed by Tensor; the head dim is contiguous. (Packed batches are
  // [total, H, d] and ignore these.)
  long long st[kTensors][3];
  // Elements each tensor spans from its base pointer (largest offset + 1),
  // and rows of lse: what the debug build's bounds checks compare against.
  long long ext[kTensors];
  long long lse_ext;
  // 1 for a call on strided dense tensors (the *_strided entry points): its
  // tensor maps are 4-D {d, L, H, B}, boxes addressed (column, row, head,
  // batch), and it runs kernel variants of their own; 0 for contiguous
  // tensors, whose maps are 3-D {d, L, B*H} addressed (column, row, unit).
  int strided;
};

#ifdef SDPA_DEBUG
__device__ __forceinline__ bool bounds_ok(bool ok, unsigned* status) {
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
}
#endif

// Element offset of row `row` of unit (b, h) in dense tensor `t`.
__host__ __device__ __forceinline__ long long dense_off(const Problem& p, int t, long long b, long long h,
                                                        long long row) {
  return b * p.st[t][0] + h * p.st[t][1] + row * p.st[t][2];
}

// Rows and keys per block of a block-sparse mask.
constexpr int kMaskBlock = 128;

struct BwdProblem {
  Problem f;          // q, k, v, o, lse as in the forward
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* delta;       // [rows] fp32 workspace: rowsum(dO * O)
  float* dq_acc;      // [rows, d] fp32 workspace (tensor-core path only)
  long long acc_rows; // rows of delta and dq_acc (debug bounds checks)
  int group;          // tensor-core kernel: units per scheduling group (set by its launcher)
};

// Tensor maps for the tensor-core kernels (built on the host by the C-ABI layer).
struct FwdMaps {
  CUtensorMap q, k, v;
  CUtensorMap mask;   // additive mask [B|1][H|1][Lq][Lk], 32 x 64 swizzled boxes (masked forward only)
};
struct BwdMaps {
  CUtensorMap q, k, v, dO;
  CUtensorMap mask;   // additive mask [B|1][H|1][Lq][Lk], 32 x 128 boxes (masked backward only)
};

// Records the message sdpa_last_error() returns on this thread; returns `code`.
int set_last_error(int code, const char* fmt, ...);

// Launchers (each in its own translation unit).
cudaError_t launch_fwd_simt(const Problem& p, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdProblem& p, cudaStream_t s);
cudaError_t launch_fwd_tc(const Problem& p, int dtype, const FwdMaps& maps, cudaStream_t s);
cudaError_t launch_bwd_prep(const BwdProblem& p, int dtype, int zero_dq_acc, cudaStream_t s);
cudaError_t launch_bwd_tc(const BwdProblem& p, int dtype, const BwdMaps& maps, cudaStream_t s);
cudaError_t launch_dq_convert(const BwdProblem& p, int dtype, cudaStream_t s);

}  // namespace sdpa
