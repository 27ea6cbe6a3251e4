// simt_f32.cu -- plain-fp32 attention kernels (FFMA + expf, no tensor cores,
// no TF32) for float32 inputs, where the 1e-5 error budget rules out reduced
// precision operands.
//
// Forward: one thread per query row streams K/V tiles through shared memory
// and keeps a running maximum m, running sum l and unnormalised output, rescaled
// whenever m grows (the online softmax that lets the FlashAttention news
// article's tiled algorithm, section "FlashAttention", stay exact). It writes
// O = acc / l and LSE = m + log l.
// Backward (recompute, same section): one kernel walks keys per query row for
// dQ, another walks queries per key row for dK and dV; both rebuild
// P_ij = exp(scale q_i.k_j - LSE_i) and dS_ij = P_ij (dO_i.v_j - D_i) with
// D_i = rowsum(dO_i * O_i) from the prep kernel.
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kRows = 128;   // query (or key) rows per block
constexpr int kTile = 32;    // rows of the other operand staged per step

struct Unit {
  int len_q, len_k;   // rows of this (batch|sequence, head)
  int b, h;           // batch (or sequence) and head
  long long tok0;     // packed: token of query row 0 / key row 0
  long long tok0k;
  long long stat;     // offset of row 0 in lse / delta
  bool bad;           // packed lengths outside their bounds
};

__device__ __forceinline__ Unit unit_of(const Problem& p, int b, int h) {
  Unit u;
  u.bad = false;
  u.b = b;
  u.h = h;
  u.tok0 = u.tok0k = 0;
  if (p.cu_seqlens == nullptr) {
    u.len_q = p.Lq;
    u.len_k = p.Lk;
    u.stat = (static_cast<long long>(b) * p.H + h) * p.Lq;
  } else {
    const int s0 = p.cu_seqlens[b], t0 = p.cu_k[b];
    u.len_q = p.cu_seqlens[b + 1] - s0;
    u.len_k = p.cu_k[b + 1] - t0;
    u.tok0 = s0;
    u.tok0k = t0;
    u.stat = static_cast<long long>(h) * p.Lq + s0;
    u.bad = u.len_q > p.max_q || u.len_k > p.Lk || (u.len_q > 0 && u.len_k <= 0);
  }
  return u;
}

// Element offset of row `row` of the unit in tensor `t`: dense at the
// tensor's strides, packed [total, H, d] on the query or key token axis.
__device__ __forceinline__ long long row_off(const Problem& p, const Unit& u, int t, long long row) {
  if (p.cu_seqlens == nullptr) return dense_off(p, t, u.b, u.h, row);
  const bool key = t == kTk || t == kTv || t == kTdk || t == kTdv;
  return ((key ? u.tok0k : u.tok0) + row) * p.H * p.d + static_cast<long long>(u.h) * p.d;
}

// Dropout factor of score (i, j) of dense unit `unit` (see Problem::dropout).
__device__ __forceinline__ float drop_factor(const Problem& p, int unit, int i, int j) {
  const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(j >> 4), static_cast<uint32_t>(i),
                                           static_cast<uint32_t>(unit), 0u),
                                p.seed_lo, p.seed_hi);
  const int b = j & 15;
  const uint32_t w = b < 8 ? (b < 4 ? r.x : r.y) : (b < 12 ? r.z : r.w);
  return ((w >> (8 * (b & 3))) & 0xffu) >= p.drop_t ? p.drop_scale : 0.f;
}

template <int DMAX>
__global__ void __launch_bounds__(kRows) fwd_f32_kernel(Problem p) {
  const int b = blockIdx.z, h = blockIdx.y;
  const Unit u = unit_of(p, b, h);
  if (u.bad) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
    return;
  }
  const int row0 = blockIdx.x * kRows;
  if (row0 >= u.len_q) return;
  const int row = row0 + threadIdx.x;
  const bool live = row < u.len_q;
  const int d = p.d;
  const float* Q = static_cast<const float*>(p.q) + row_off(p, u, kTq, row);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);

  __shared__ float sk[kTile][DMAX];
  __shared__ float sv[kTile][DMAX];

  float qr[DMAX], acc[DMAX];
#pragma unroll
  for (int c = 0; c < DMAX; ++c) {
    qr[c] = (live && c < d) ? Q[c] : 0.f;
    acc[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const unsigned char* mrow = p.bmask ? p.bmask + b * p.bm_sb + h * p.bm_sh + (row / kMaskBlock) * p.bm_sq : nullptr;
  const float* arow = p.amask ? static_cast<const float*>(p.amask) + b * p.am_sb + h * p.am_sh + row * p.am_sq : nullptr;
  int kend = u.len_k;
  if (p.causal) kend = min(kend, min(row0 + kRows, u.len_q));
  for (int kb = 0; kb < kend; kb += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * DMAX; e += kRows) {
      const int r = e / DMAX, c = e % DMAX;
      const bool ok = (kb + r < u.len_k) && c < d;
      sk[r][c] = ok ? K[row_off(p, u, kTk, kb + r) + c] : 0.f;
      sv[r][c] = ok ? V[row_off(p, u, kTv, kb + r) + c] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    for (int jj = 0; jj < kTile; ++jj) {
      const int key = kb + jj;
      if (key >= u.len_k || (p.causal && key > row)) break;
      if (mrow && !mrow[key / kMaskBlock]) continue;
      const float bias = arow ? arow[key] : 0.f;
      if (bias == -INFINITY) continue;
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < DMAX; ++c) s = fmaf(qr[c], sk[jj][c], s);
      s = s * p.scale + bias;
      if (s > m) {
        const float corr = expf(m - s);
        l *= corr;
#pragma unroll
        for (int c = 0; c < DMAX; ++c) acc[c] *= corr;
        m = s;
      }
      const float e = expf(s - m);
      l += e;
      const float ez = p.dropout ? e * drop_factor(p, b * p.H + h, row, key) : e;   // P . V sees dropout
#pragma unroll
      for (int c = 0; c < DMAX; ++c) acc[c] = fmaf(ez, sv[jj][c], acc[c]);
    }
  }
  if (!live) return;
  const long long oo = row_off(p, u, kTo, row);
  if (!SDPA_CHECK(oo + d <= p.ext[kTo] && u.stat + row < p.lse_ext, p.status)) return;
  float* O = static_cast<float*>(p.o) + oo;
  // a row with no visible key (block-sparse only) gets O = 0 and LSE = -inf
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < DMAX; ++c)
    if (c < d) O[c] = acc[c] * inv;
  p.lse[u.stat + row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// dQ_i = scale * sum_j P_ij (dO_i.v_j - D_i) k_j
template <int DMAX>
__global__ void __launch_bounds__(kRows) bwd_dq_f32_kernel(BwdProblem bp) {
  const Problem& p = bp.f;
  const int b = blockIdx.z, h = blockIdx.y;
  const Unit u = unit_of(p, b, h);
  if (u.bad) {   // lengths outside their bounds: reported, nothing written
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
    return;
  }
  const int row0 = blockIdx.x * kRows;
  if (row0 >= u.len_q) return;
  const int row = row0 + threadIdx.x;
  const bool live = row < u.len_q;
  const int d = p.d;
  const float* Q = static_cast<const float*>(p.q) + row_off(p, u, kTq, row);
  const float* dO = static_cast<const float*>(bp.dO) + row_off(p, u, kTdo, row);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);

  __shared__ float sk[kTile][DMAX];
  __shared__ float sv[kTile][DMAX];
  float qr[DMAX], dor[DMAX], dq[DMAX];
#pragma unroll
  for (int c = 0; c < DMAX; ++c) {
    qr[c] = (live && c < d) ? Q[c] : 0.f;
    dor[c] = (live && c < d) ? dO[c] : 0.f;
    dq[c] = 0.f;
  }
  const float lse = live ? p.lse[u.stat + row] : 0.f;
  const float D = live ? bp.delta[u.stat + row] : 0.f;
  const unsigned char* mrow = p.bmask ? p.bmask + b * p.bm_sb + h * p.bm_sh + (row / kMaskBlock) * p.bm_sq : nullptr;
  const float* arow = p.amask ? static_cast<const float*>(p.amask) + b * p.am_sb + h * p.am_sh + row * p.am_sq : nullptr;
  int kend = u.len_k;
  if (p.causal) kend = min(kend, min(row0 + kRows, u.len_q));
  for (int kb = 0; kb < kend; kb += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * DMAX; e += kRows) {
      const int r = e / DMAX, c = e % DMAX;
      const bool ok = (kb + r < u.len_k) && c < d;
      sk[r][c] = ok ? K[row_off(p, u, kTk, kb + r) + c] : 0.f;
      sv[r][c] = ok ? V[row_off(p, u, kTv, kb + r) + c] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    for (int jj = 0; jj < kTile; ++jj) {
      const int key = kb + jj;
      if (key >= u.len_k || (p.causal && key > row)) break;
      if (mrow && !mrow[key / kMaskBlock]) continue;
      const float bias = arow ? arow[key] : 0.f;
      if (bias == -INFINITY) continue;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < DMAX; ++c) {
        s = fmaf(qr[c], sk[jj][c], s);
        dp = fmaf(dor[c], sv[jj][c], dp);
      }
      const float pr = expf(s * p.scale + bias - lse);
      const float z = p.dropout ? drop_factor(p, b * p.H + h, row, key) : 1.f;
      const float ds = pr * (dp * z - D);
#pragma unroll
      for (int c = 0; c < DMAX; ++c) dq[c] = fmaf(ds, sk[jj][c], dq[c]);
    }
  }
  if (!live) return;
  const long long qo = row_off(p, u, kTdq, row);
  if (!SDPA_CHECK(qo + d <= p.ext[kTdq], p.status)) return;
  float* dQ = static_cast<float*>(bp.dq) + qo;
#pragma unroll
  for (int c = 0; c < DMAX; ++c)
    if (c < d) dQ[c] = dq[c] * p.scale;
}

// dV_j = sum_i P_ij dO_i ; dK_j = scale * sum_i P_ij (dO_i.v_j - D_i) q_i
template <int DMAX>
__global__ void __launch_bounds__(kRows) bwd_dkdv_f32_kernel(BwdProblem bp) {
  const Problem& p = bp.f;
  const int b = blockIdx.z, h = blockIdx.y;
  const Unit u = unit_of(p, b, h);
  if (u.bad) return;   // reported by the dQ kernel
  const int key0 = blockIdx.x * kRows;
  if (key0 >= u.len_k) return;
  const int key = key0 + threadIdx.x;
  const bool live = key < u.len_k;
  const int d = p.d;
  const float* Q = static_cast<const float*>(p.q);
  const float* dO = static_cast<const float*>(bp.dO);
  const float* K = static_cast<const float*>(p.k) + row_off(p, u, kTk, key);
  const float* V = static_cast<const float*>(p.v) + row_off(p, u, kTv, key);

  __shared__ float sq[kTile][DMAX];
  __shared__ float sdo[kTile][DMAX];
  __shared__ float slse[kTile], sD[kTile];
  float kr[DMAX], vr[DMAX], dk[DMAX], dv[DMAX];
#pragma unroll
  for (int c = 0; c < DMAX; ++c) {
    kr[c] = (live && c < d) ? K[c] : 0.f;
    vr[c] = (live && c < d) ? V[c] : 0.f;
    dk[c] = 0.f;
    dv[c] = 0.f;
  }
  const int qstart = p.causal ? key0 : 0;
  for (int qb = qstart; qb < u.len_q; qb += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * DMAX; e += kRows) {
      const int r = e / DMAX, c = e % DMAX;
      const bool ok = (qb + r < u.len_q) && c < d;
      sq[r][c] = ok ? Q[row_off(p, u, kTq, qb + r) + c] : 0.f;
      sdo[r][c] = ok ? dO[row_off(p, u, kTdo, qb + r) + c] : 0.f;
    }
    if (threadIdx.x < kTile) {
      const int r = qb + threadIdx.x;
      slse[threadIdx.x] = r < u.len_q ? p.lse[u.stat + r] : 0.f;
      sD[threadIdx.x] = r < u.len_q ? bp.delta[u.stat + r] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    for (int ii = 0; ii < kTile; ++ii) {
      const int qi = qb + ii;
      if (qi >= u.len_q) break;
      if (p.causal && key > qi) continue;
      if (p.bmask && !p.bmask[b * p.bm_sb + h * p.bm_sh + (qi / kMaskBlock) * p.bm_sq + key / kMaskBlock]) continue;
      const float bias =
          p.amask ? static_cast<const float*>(p.amask)[b * p.am_sb + h * p.am_sh + qi * p.am_sq + key] : 0.f;
      if (bias == -INFINITY) continue;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < DMAX; ++c) {
        s = fmaf(sq[ii][c], kr[c], s);
        dp = fmaf(sdo[ii][c], vr[c], dp);
      }
      const float pr = expf(s * p.scale + bias - slse[ii]);
      const float z = p.dropout ? drop_factor(p, b * p.H + h, qi, key) : 1.f;
      const float ds = pr * (dp * z - sD[ii]);
#pragma unroll
      for (int c = 0; c < DMAX; ++c) {
        dv[c] = fmaf(pr * z, sdo[ii][c], dv[c]);
        dk[c] = fmaf(ds, sq[ii][c], dk[c]);
      }
    }
  }
  if (!live) return;
  const long long ko = row_off(p, u, kTdk, key), vo = row_off(p, u, kTdv, key);
  if (!SDPA_CHECK(ko + d <= p.ext[kTdk] && vo + d <= p.ext[kTdv], p.status)) return;
  float* dK = static_cast<float*>(bp.dk) + ko;
  float* dV = static_cast<float*>(bp.dv) + vo;
#pragma unroll
  for (int c = 0; c < DMAX; ++c) {
    if (c < d) {
      dK[c] = dk[c] * p.scale;
      dV[c] = dv[c];
    }
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& p, cudaStream_t s) {
  const bool packed = p.cu_seqlens != nullptr;
  const int rows = packed ? p.max_q : p.Lq;  // packed: max_q bounds every query length
  dim3 grid((rows + kRows - 1) / kRows, p.H, p.B);
  if (grid.x == 0) return cudaSuccess;
  if (p.d <= 32) fwd_f32_kernel<32><<<grid, kRows, 0, s>>>(p);
  else if (p.d <= 64) fwd_f32_kernel<64><<<grid, kRows, 0, s>>>(p);
  else fwd_f32_kernel<128><<<grid, kRows, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdProblem& bp, cudaStream_t s) {
  const Problem& p = bp.f;
  const bool packed = p.cu_seqlens != nullptr;
  const int rq = packed ? p.max_q : p.Lq;  // packed: bounds on the query and key lengths
  const int rk = p.Lk;
  dim3 gq((rq + kRows - 1) / kRows, p.H, p.B), gk((rk + kRows - 1) / kRows, p.H, p.B);
  if (p.d <= 32) {
    if (gq.x) bwd_dq_f32_kernel<32><<<gq, kRows, 0, s>>>(bp);
    if (gk.x) bwd_dkdv_f32_kernel<32><<<gk, kRows, 0, s>>>(bp);
  } else if (p.d <= 64) {
    if (gq.x) bwd_dq_f32_kernel<64><<<gq, kRows, 0, s>>>(bp);
    if (gk.x) bwd_dkdv_f32_kernel<64><<<gk, kRows, 0, s>>>(bp);
  } else {
    if (gq.x) bwd_dq_f32_kernel<128><<<gq, kRows, 0, s>>>(bp);
    if (gk.x) bwd_dkdv_f32_kernel<128><<<gk, kRows, 0, s>>>(bp);
  }
  return cudaGetLastError();
}

}  // namespace sdpa
