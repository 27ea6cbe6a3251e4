// api.cu -- the C ABI declared in include/sdpa.h: argument checks, tensor-map
// construction, the device status word, and dispatch to the kernels.
// All checks run on the host before anything is launched; no call allocates.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "sdpa.h"

namespace sdpa {
namespace {

thread_local std::string g_last_error;
int g_debug_flags = 0;

// Kernel timing aid: caller-owned CUDA events recorded on the call's stream
// around the main attention kernel of the forward ([0]) and backward ([1]).
cudaEvent_t g_trace_begin[2] = {nullptr, nullptr};
cudaEvent_t g_trace_end[2] = {nullptr, nullptr};

cudaError_t trace_mark(const cudaEvent_t* evs, int which, cudaStream_t s) {
  return evs[which] ? cudaEventRecord(evs[which], s) : cudaSuccess;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(SDPA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// One status word per device that loads the library; kernels OR bits into it.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {nullptr};

int status_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SDPA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    g_status_ptr[dev] = static_cast<unsigned*>(ptr);
  }
  *out = g_status_ptr[dev];
  return SDPA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return SDPA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return SDPA_OK;
}

// 4-D tiled map over 16-bit elements: dims {d, n1, n2, n3} with the byte
// strides of dims 1..3, box {box0, box1, 1, 1} or {box0, 1, box2, 1}. A
// dimension of size 1 takes a harmless stride (its coordinate is always 0).
int make_map4(CUtensorMap* m, const void* base, int dtype, uint64_t d, uint64_t n1, uint64_t n2, uint64_t n3,
              uint64_t s1, uint64_t s2, uint64_t s3, uint32_t box0, uint32_t box1, uint32_t box2) {
  const uint64_t fill = std::max<uint64_t>({16, n1 * s1, n2 * s2});
  if (n1 == 1) s1 = (s1 % 16 == 0 && s1 > 0) ? s1 : (d * 2 + 15) / 16 * 16;
  if (n2 == 1) s2 = (s2 % 16 == 0 && s2 > 0) ? s2 : (fill + 15) / 16 * 16;
  if (n3 == 1) s3 = (s3 % 16 == 0 && s3 > 0) ? s3 : (fill + 15) / 16 * 16;
  const cuuint64_t dims[4] = {d, n1, n2, n3};
  const cuuint64_t strides[3] = {s1, s2, s3};
  const cuuint32_t box[4] = {box0, box1, box2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = box0 * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return SDPA_OK;
}

// 3-D tiled map over 16-bit elements: dims {d, n1, n2}, byte strides of
// dims 1 and 2, box {box0, box1, box2}.
int make_map3(CUtensorMap* m, const void* base, int dtype, uint64_t d, uint64_t n1, uint64_t n2, uint64_t s1,
              uint64_t s2, uint32_t box0, uint32_t box1, uint32_t box2) {
  const cuuint64_t dims[3] = {d, n1, n2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = box0 * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return SDPA_OK;
}

// Map for a q/k/v-like tensor, tiled in `box_rows`-row boxes of 64 (d >= 64)
// or 32 (d = 32) columns. Contiguous dense: dims {d, rows, B*H}, boxes at
// (column, row, unit). Strided dense: dims {d, rows, H, B} at the tensor's
// element strides `st` = (batch, head, row), boxes at (column, row, head,
// batch). Packed [total, H, d]: dims {d, H, total}, boxes at (column, head,
// token).
int make_operand_map(CUtensorMap* m, const void* base, int dtype, bool packed, int B, int H, int rows, int d,
                     const long long* st, int strided, uint32_t box_rows = 128) {
  const uint32_t blk = d >= 64 ? 64 : static_cast<uint32_t>(d);
  const uint64_t es = 2;
  if (packed) return make_map3(m, base, dtype, d, H, rows, d * es, static_cast<uint64_t>(H) * d * es, blk, 1, box_rows);
  if (strided) return make_map4(m, base, dtype, d, rows, H, B, st[2] * es, st[1] * es, st[0] * es, blk, box_rows, 1);
  return make_map3(m, base, dtype, d, rows, static_cast<uint64_t>(B) * H, d * es, static_cast<uint64_t>(rows) * d * es,
                   blk, box_rows, 1);
}

// Map over an additive mask with element strides (sb, sh, sq): dims {Lk, Lq,
// H, B}, a batch or head stride of 0 (broadcast) becomes a dimension of size
// 1; boxes of `box_rows` query rows x `box_keys` keys, 128-byte swizzled when
// a box row is 128 bytes (64 keys), else unswizzled. Reads past Lk or Lq fill
// zeros, so no padding of the rows is read.
int make_mask_map(CUtensorMap* m, const void* base, int dtype, int B, int H, int Lq, int Lk, long long sb, long long sh,
                  long long sq, uint32_t box_keys, uint32_t box_rows) {
  const uint64_t es = 2;
  const uint64_t nh = sh ? static_cast<uint64_t>(H) : 1, nb = sb ? static_cast<uint64_t>(B) : 1;
  const uint64_t rs = static_cast<uint64_t>(sq) * es;
  const uint64_t hs = sh ? static_cast<uint64_t>(sh) * es : rs * static_cast<uint64_t>(Lq);
  const uint64_t bs = sb ? static_cast<uint64_t>(sb) * es : hs * nh;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Lk), static_cast<cuuint64_t>(Lq), nh, nb};
  const cuuint64_t strides[3] = {rs, hs, bs};
  const cuuint32_t box[4] = {box_keys, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = box_keys * es == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the attention mask (CUresult %d)", static_cast<int>(r));
  return SDPA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int set_last_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

}  // namespace sdpa

using namespace sdpa;

namespace {

// Sizes of one call. Dense: cu_q = cu_k = NULL, [B,H,Lq,d] / [B,H,Lk,d].
// Packed: B sequences; queries on `total_q` rows through cu_q, keys on
// `total_k` rows through cu_k; max_q / max_k bound the lengths.
struct Shape {
  int B, H, total_q, total_k, max_q, max_k, d;
  const int* cu_q;
  const int* cu_k;
  bool packed() const { return cu_q != nullptr; }
};

// Block-sparse mask (dense layout only): 0/1 per (128-query, 128-key) tile.
struct BlockMask {
  const unsigned char* m;
  long long sb, sh;
  int sq;
};

// Additive mask (dense layout only), in the input dtype, keys contiguous.
struct AddMask {
  const void* m;
  long long sb, sh, sq;
};

int check_addmask(const Shape& sh, const AddMask& am, int dtype) {
  if (am.m == nullptr) return fail(SDPA_ERR_ARG, "attention mask pointer is NULL");
  if (am.sb < 0 || am.sh < 0 || am.sq < sh.total_k)
    return fail(SDPA_ERR_ARG, "attention mask strides must be non-negative and the row stride at least Lk = %d", sh.total_k);
  if (dtype != SDPA_F32) {
    // the tensor-core kernels read the mask with TMA: 16-byte aligned base and strides
    const long long lk8 = (sh.total_k + 7) / 8 * 8;
    if (!aligned16(am.m) || am.sq % 8 != 0 || am.sb % 8 != 0 || am.sh % 8 != 0 || am.sq < lk8)
      return fail(SDPA_ERR_ARG, "fp16/bf16 attention masks need a 16-byte aligned base, strides that are multiples of 8 "
                                "elements and a row stride of at least %lld", lk8);
  }
  return SDPA_OK;
}

// Dropout (dense layout only).
struct Dropout {
  float p;
  unsigned long long seed;
};

// Longest query axis a block-sparse backward accepts: its CTAs list their
// active query steps (up to 2048 of 64 or 128 rows) in shared memory.
constexpr int kMaxSparseLq = 131072;

int check_mask(const Shape& sh, const BlockMask& bm, bool backward) {
  if (bm.m == nullptr) return fail(SDPA_ERR_ARG, "block mask pointer is NULL");
  if (sh.packed()) return fail(SDPA_ERR_UNSUPPORTED, "block masks apply to the dense layout only");
  const int nkb = (sh.total_k + kMaskBlock - 1) / kMaskBlock;
  if (bm.sb < 0 || bm.sh < 0 || bm.sq < nkb)
    return fail(SDPA_ERR_ARG, "block mask strides must be non-negative and the row stride at least %d (got %lld, %lld, %d)",
                nkb, bm.sb, bm.sh, bm.sq);
  if (backward && sh.total_q > kMaxSparseLq)
    return fail(SDPA_ERR_UNSUPPORTED, "block-sparse backward supports Lq <= %d (got %d)", kMaxSparseLq, sh.total_q);
  return SDPA_OK;
}

int check_shape(const Shape& sh, float scale, int is_causal, int dtype, bool* noop) {
  *noop = false;
  if (dtype != SDPA_F32 && dtype != SDPA_F16 && dtype != SDPA_BF16) return fail(SDPA_ERR_ARG, "unknown dtype %d", dtype);
  if (sh.B < 0 || sh.H < 0 || sh.total_q < 0 || sh.total_k < 0 || sh.max_q < 0 || sh.max_k < 0 || sh.d <= 0)
    return fail(SDPA_ERR_ARG, "sizes must be non-negative and d positive (B=%d H=%d Lq=%d Lk=%d d=%d)", sh.B, sh.H,
                sh.total_q, sh.total_k, sh.d);
  if (!std::isfinite(scale)) return fail(SDPA_ERR_ARG, "scale must be finite");
  if (is_causal != 0 && is_causal != 1) return fail(SDPA_ERR_ARG, "is_causal must be 0 or 1");
  if (dtype == SDPA_F32) {
    if (sh.d > 128) return fail(SDPA_ERR_UNSUPPORTED, "float32 path supports d <= 128 (got %d)", sh.d);
  } else if (sh.d != 32 && sh.d != 64 && sh.d != 128) {
    return fail(SDPA_ERR_UNSUPPORTED, "fp16/bf16 path supports d in {32, 64, 128} (got %d)", sh.d);
  }
  if (sh.packed() && sh.cu_k == nullptr) return fail(SDPA_ERR_ARG, "key offsets missing");
  if (sh.B == 0 || sh.H == 0 || sh.total_q == 0 || (sh.packed() && sh.max_q == 0)) {
    *noop = true;  // no query rows
    return SDPA_OK;
  }
  if (sh.max_k == 0 || sh.total_k == 0) return fail(SDPA_ERR_ARG, "no keys for %d query rows: softmax over no keys", sh.total_q);
  return SDPA_OK;
}

int check_tensors(const void* q, const void* k, const void* v, const void* o, const float* lse, int dtype) {
  if (!q || !k || !v || !o || !lse) return fail(SDPA_ERR_ARG, "null tensor pointer");
  if (dtype != SDPA_F32 && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o)))
    return fail(SDPA_ERR_ARG, "fp16/bf16 tensors must be 16-byte aligned");
  return SDPA_OK;
}

void fill_problem(Problem& p, const Shape& sh, const void* q, const void* k, const void* v, const void* o,
                  const float* lse, float scale, int is_causal, const BlockMask& bm,
                  const AddMask& am = AddMask{nullptr, 0, 0, 0}, const Dropout& dr = Dropout{0.f, 0ull}) {
  // p is used as a multiple of 1/256: bytes below t = round(256 p) drop
  const int t = std::min(static_cast<int>(std::lround(dr.p * 256.0f)), 255);
  p.dropout = t > 0 ? 1 : 0;
  p.drop_t = static_cast<unsigned>(t);
  p.drop_scale = 256.0f / static_cast<float>(256 - t);
  p.seed_lo = static_cast<unsigned>(dr.seed & 0xffffffffull);
  p.seed_hi = static_cast<unsigned>(dr.seed >> 32);
  p.amask = am.m;
  p.am_sb = am.sb;
  p.am_sh = am.sh;
  p.am_sq = am.sq;
  p.bmask = bm.m;
  p.bm_sb = bm.sb;
  p.bm_sh = bm.sh;
  p.bm_sq = bm.sq;
  p.q = q; p.k = k; p.v = v; p.o = const_cast<void*>(o); p.lse = const_cast<float*>(lse);
  p.B = sh.B; p.H = sh.H; p.d = sh.d;
  p.scale = scale; p.causal = is_causal;
  p.cu_seqlens = sh.cu_q;
  p.cu_k = sh.cu_k;
  p.Lq = sh.total_q;
  // dense: Lk is the key length of every unit; packed: the bound on it
  p.Lk = sh.packed() ? sh.max_k : sh.total_k;
  p.total_k = sh.total_k;
  p.max_q = sh.packed() ? sh.max_q : sh.total_q;
  p.debug = g_debug_flags;
  // dense tensors contiguous unless the call gives strides
  for (int t = 0; t < kTensors; ++t) {
    const bool key = t == kTk || t == kTv || t == kTdk || t == kTdv;
    const long long rows = key ? sh.total_k : sh.total_q;
    p.st[t][2] = sh.d;
    p.st[t][1] = rows * sh.d;
    p.st[t][0] = static_cast<long long>(sh.H) * rows * sh.d;
  }
}

// Strides of a strided call: `n` tensors in Tensor order, (batch, head, row)
// each, in elements. Every stride of a dimension longer than 1 must be
// positive; fp16 / bf16 strides must be multiples of 8 elements (16 bytes:
// the tensor-core kernels read with TMA and store 16-byte vectors).
int check_strides(const Shape& sh, const long long* strides, int n, int dtype) {
  if (strides == nullptr) return fail(SDPA_ERR_ARG, "stride array is NULL");
  static const char* names[kTensors] = {"q", "k", "v", "o", "dO", "dq", "dk", "dv"};
  for (int t = 0; t < n; ++t) {
    const bool key = t == kTk || t == kTv || t == kTdk || t == kTdv;
    const long long ext[3] = {sh.B, sh.H, key ? sh.total_k : sh.total_q};
    for (int i = 0; i < 3; ++i) {
      const long long v = strides[3 * t + i];
      if (v < 0 || (v == 0 && ext[i] > 1))
        return fail(SDPA_ERR_ARG, "stride %d of %s is %lld: strides must be positive", i, names[t], v);
      if (dtype != SDPA_F32 && v % 8 != 0)
        return fail(SDPA_ERR_ARG, "stride %d of %s is %lld: fp16/bf16 strides must be multiples of 8 elements", i,
                    names[t], v);
    }
  }
  return SDPA_OK;
}

void set_strides(Problem& p, const long long* strides, int n) {
  if (strides == nullptr) return;
  p.strided = 1;
  for (int t = 0; t < n; ++t)
    for (int i = 0; i < 3; ++i) p.st[t][i] = strides[3 * t + i];
}

// Elements each tensor spans (largest element offset + 1) and rows of lse,
// for the debug build's bounds checks; after set_strides.
void set_extents(Problem& p, const Shape& sh) {
  for (int t = 0; t < kTensors; ++t) {
    const bool key = t == kTk || t == kTv || t == kTdk || t == kTdv;
    const long long rows = key ? sh.total_k : sh.total_q;
    if (sh.packed()) p.ext[t] = rows * sh.H * sh.d;
    else if (sh.B == 0 || sh.H == 0 || rows == 0) p.ext[t] = 0;
    else p.ext[t] = (sh.B - 1) * p.st[t][0] + (sh.H - 1) * p.st[t][1] + (rows - 1) * p.st[t][2] + sh.d;
  }
  p.lse_ext = static_cast<long long>(sh.packed() ? 1 : sh.B) * sh.H * sh.total_q;
  if (p.debug & kDebugShortO) p.ext[kTo] -= sh.d;
}

int run_fwd(const Shape& sh, const void* q, const void* k, const void* v, void* o, float* lse, float scale,
            int is_causal, int dtype, void* stream, const BlockMask& bm = BlockMask{nullptr, 0, 0, 0}, bool sparse = false,
            const AddMask& am = AddMask{nullptr, 0, 0, 0}, bool masked = false,
            const Dropout& dr = Dropout{0.f, 0ull}, const long long* strides = nullptr) {
  g_last_error.clear();
  bool noop = false;
  int rc = check_shape(sh, scale, is_causal, dtype, &noop);
  if (rc != SDPA_OK || noop) return rc;
  if ((rc = check_tensors(q, k, v, o, lse, dtype)) != SDPA_OK) return rc;
  if (sparse && (rc = check_mask(sh, bm, false)) != SDPA_OK) return rc;
  if (masked && (rc = check_addmask(sh, am, dtype)) != SDPA_OK) return rc;
  if (!(dr.p >= 0.f && dr.p < 1.f)) return fail(SDPA_ERR_ARG, "dropout probability must be in [0, 1) (got %g)", dr.p);
  if (strides != nullptr && (rc = check_strides(sh, strides, 4, dtype)) != SDPA_OK) return rc;
  Problem p{};
  fill_problem(p, sh, q, k, v, o, lse, scale, is_causal, bm, am, dr);
  set_strides(p, strides, 4);
  set_extents(p, sh);
  rc = status_ptr(&p.status);
  if (rc != SDPA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SDPA_F32) {
    if ((e = trace_mark(g_trace_begin, 0, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
    e = launch_fwd_simt(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "forward (fp32) launch");
    if ((e = trace_mark(g_trace_end, 0, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
    return SDPA_OK;
  }
  rc = get_encoder();
  if (rc != SDPA_OK) return rc;
  const bool packed = sh.packed();
  FwdMaps maps{};
  if ((rc = make_operand_map(&maps.q, q, dtype, packed, sh.B, sh.H, sh.total_q, sh.d, p.st[kTq], p.strided)) != SDPA_OK)
    return rc;
  if ((rc = make_operand_map(&maps.k, k, dtype, packed, sh.B, sh.H, sh.total_k, sh.d, p.st[kTk], p.strided)) != SDPA_OK)
    return rc;
  if ((rc = make_operand_map(&maps.v, v, dtype, packed, sh.B, sh.H, sh.total_k, sh.d, p.st[kTv], p.strided)) != SDPA_OK)
    return rc;
  // additive mask: each softmax warp loads its 32 rows of a 128-key block as two 64-key boxes
  if (masked &&
      (rc = make_mask_map(&maps.mask, am.m, dtype, sh.B, sh.H, sh.total_q, sh.total_k, am.sb, am.sh, am.sq, 64, 32)) !=
          SDPA_OK)
    return rc;
  if ((e = trace_mark(g_trace_begin, 0, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
  e = launch_fwd_tc(p, dtype, maps, s);
  if (e != cudaSuccess) return cuda_fail(e, "forward (tensor-core) launch");
  if ((e = trace_mark(g_trace_end, 0, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
  return SDPA_OK;
}

int run_bwd(const Shape& sh, const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dO, void* dq, void* dk, void* dv, float scale, int is_causal, int dtype, void* workspace,
            size_t workspace_bytes, void* stream, const BlockMask& bm = BlockMask{nullptr, 0, 0, 0},
            bool sparse = false, const AddMask& am = AddMask{nullptr, 0, 0, 0}, bool masked = false,
            const Dropout& dr = Dropout{0.f, 0ull}, const long long* strides = nullptr) {
  g_last_error.clear();
  bool noop = false;
  int rc = check_shape(sh, scale, is_causal, dtype, &noop);
  if (rc != SDPA_OK || noop) return rc;
  if ((rc = check_tensors(q, k, v, o, lse, dtype)) != SDPA_OK) return rc;
  if (sparse && (rc = check_mask(sh, bm, true)) != SDPA_OK) return rc;
  if (masked && (rc = check_addmask(sh, am, dtype)) != SDPA_OK) return rc;
  if (!(dr.p >= 0.f && dr.p < 1.f)) return fail(SDPA_ERR_ARG, "dropout probability must be in [0, 1) (got %g)", dr.p);
  if (!dO || !dq || !dk || !dv) return fail(SDPA_ERR_ARG, "null gradient pointer");
  if (dtype != SDPA_F32 && !(aligned16(dO) && aligned16(dq) && aligned16(dk) && aligned16(dv)))
    return fail(SDPA_ERR_ARG, "fp16/bf16 gradients must be 16-byte aligned");
  const bool packed = sh.packed();
  // packed: the row statistics and dQ accumulator cover the total query rows
  const int nb = packed ? 1 : sh.B;
  const size_t need = sdpa_bwd_workspace_size(nb, sh.H, sh.total_q, sh.d, dtype);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace == nullptr ? 0 : workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(SDPA_ERR_ARG, "workspace must be 256-byte aligned");

  if (strides != nullptr && (rc = check_strides(sh, strides, kTensors, dtype)) != SDPA_OK) return rc;
  BwdProblem bp{};
  Problem& p = bp.f;
  fill_problem(p, sh, q, k, v, o, lse, scale, is_causal, bm, am, dr);
  set_strides(p, strides, kTensors);
  set_extents(p, sh);
  rc = status_ptr(&p.status);
  if (rc != SDPA_OK) return rc;
  bp.dO = dO; bp.dq = dq; bp.dk = dk; bp.dv = dv;
  const size_t rows = static_cast<size_t>(nb) * sh.H * sh.total_q;
  bp.acc_rows = static_cast<long long>(rows);
  bp.delta = static_cast<float*>(workspace);
  bp.dq_acc = dtype == SDPA_F32 ? nullptr
                                : reinterpret_cast<float*>(static_cast<char*>(workspace) + (rows * 4 + 255) / 256 * 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_prep(bp, dtype, dtype == SDPA_F32 ? 0 : 1, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward prep launch");
  if (dtype == SDPA_F32) {
    if ((e = trace_mark(g_trace_begin, 1, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
    e = launch_bwd_simt(bp, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward (fp32) launch");
    if ((e = trace_mark(g_trace_end, 1, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
    return SDPA_OK;
  }
  rc = get_encoder();
  if (rc != SDPA_OK) return rc;
  BwdMaps maps{};
  const uint32_t bq = sh.d == 128 ? 64 : 128;  // query rows per backward step
  if ((rc = make_operand_map(&maps.q, q, dtype, packed, sh.B, sh.H, sh.total_q, sh.d, p.st[kTq], p.strided, bq)) !=
      SDPA_OK)
    return rc;
  if ((rc = make_operand_map(&maps.k, k, dtype, packed, sh.B, sh.H, sh.total_k, sh.d, p.st[kTk], p.strided)) != SDPA_OK)
    return rc;
  if ((rc = make_operand_map(&maps.v, v, dtype, packed, sh.B, sh.H, sh.total_k, sh.d, p.st[kTv], p.strided)) != SDPA_OK)
    return rc;
  if ((rc = make_operand_map(&maps.dO, dO, dtype, packed, sh.B, sh.H, sh.total_q, sh.d, p.st[kTdo], p.strided, bq)) !=
      SDPA_OK)
    return rc;
  if (masked &&
      (rc = make_mask_map(&maps.mask, am.m, dtype, sh.B, sh.H, sh.total_q, sh.total_k, am.sb, am.sh, am.sq, 128, 32)) !=
          SDPA_OK)
    return rc;
  if ((e = trace_mark(g_trace_begin, 1, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
  e = launch_bwd_tc(bp, dtype, maps, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward (tensor-core) launch");
  if ((e = trace_mark(g_trace_end, 1, s)) != cudaSuccess) return cuda_fail(e, "recording the trace event");
  e = launch_dq_convert(bp, dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "dQ convert launch");
  return SDPA_OK;
}

// Dense, or packed self-attention (one offset array for queries and keys;
// Lq = total tokens, Lk = max_seqlen).
Shape self_shape(int B, int H, int Lq, int Lk, int d, const int* cu) {
  if (cu == nullptr) return Shape{B, H, Lq, Lk, Lq, Lk, d, nullptr, nullptr};
  return Shape{B, H, Lq, Lq, Lk, Lk, d, cu, cu};
}

}  // namespace

extern "C" int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Lq, int Lk,
                        int d, float scale, int is_causal, const int* cu_seqlens, int dtype, void* stream) {
  return run_fwd(self_shape(B, H, Lq, Lk, d, cu_seqlens), q, k, v, o, lse, scale, is_causal, dtype, stream);
}

extern "C" int sdpa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int Lq, int Lk, int d, float scale, int is_causal, const long long* strides,
                                int dtype, void* stream) {
  g_last_error.clear();
  if (strides == nullptr) return fail(SDPA_ERR_ARG, "stride array is NULL");
  return run_fwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, scale, is_causal, dtype, stream,
                 BlockMask{nullptr, 0, 0, 0}, false, AddMask{nullptr, 0, 0, 0}, false, Dropout{0.f, 0ull}, strides);
}

extern "C" int sdpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int nseq, int H,
                               int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, float scale,
                               int is_causal, const int* cu_seqlens_q, const int* cu_seqlens_k, int dtype,
                               void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) {
    g_last_error.clear();
    return fail(SDPA_ERR_ARG, "sdpa_fwd_varlen needs both offset arrays");
  }
  const Shape sh{nseq, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d, cu_seqlens_q, cu_seqlens_k};
  return run_fwd(sh, q, k, v, o, lse, scale, is_causal, dtype, stream);
}

extern "C" size_t sdpa_bwd_workspace_size(int B, int H, int Lq, int d, int dtype) {
  if (B <= 0 || H <= 0 || Lq <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Lq;
  const size_t delta = (rows * sizeof(float) + 255) / 256 * 256;
  if (dtype == SDPA_F32) return delta;
  return delta + rows * d * sizeof(float);
}

extern "C" int sdpa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                        const int* cu_seqlens, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return run_bwd(self_shape(B, H, Lq, Lk, d, cu_seqlens), q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype,
                 workspace, workspace_bytes, stream);
}

extern "C" int sdpa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                                float scale, int is_causal, const long long* strides, int dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  if (strides == nullptr) return fail(SDPA_ERR_ARG, "stride array is NULL");
  return run_bwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype,
                 workspace, workspace_bytes, stream, BlockMask{nullptr, 0, 0, 0}, false, AddMask{nullptr, 0, 0, 0},
                 false, Dropout{0.f, 0ull}, strides);
}

extern "C" int sdpa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dO, void* dq, void* dk, void* dv, int nseq, int H, int total_q, int total_k,
                               int max_seqlen_q, int max_seqlen_k, int d, float scale, int is_causal,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) {
    g_last_error.clear();
    return fail(SDPA_ERR_ARG, "sdpa_bwd_varlen needs both offset arrays");
  }
  const Shape sh{nseq, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d, cu_seqlens_q, cu_seqlens_k};
  return run_bwd(sh, q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype, workspace, workspace_bytes, stream);
}

extern "C" int sdpa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int Lq, int Lk, int d, float scale, int is_causal,
                                    const unsigned char* block_mask, long long mask_stride_b,
                                    long long mask_stride_h, int mask_stride_row, int dtype, void* stream) {
  const BlockMask bm{block_mask, mask_stride_b, mask_stride_h, mask_stride_row};
  return run_fwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, scale, is_causal, dtype, stream, bm, true);
}

extern "C" int sdpa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                                    float scale, int is_causal, const unsigned char* block_mask,
                                    long long mask_stride_b, long long mask_stride_h, int mask_stride_row,
                                    int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  const BlockMask bm{block_mask, mask_stride_b, mask_stride_h, mask_stride_row};
  return run_bwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype,
                 workspace, workspace_bytes, stream, bm, true);
}

extern "C" int sdpa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Lq,
                               int Lk, int d, float scale, int is_causal, const void* attn_mask,
                               long long mask_stride_b, long long mask_stride_h, long long mask_stride_row, int dtype,
                               void* stream) {
  const AddMask am{attn_mask, mask_stride_b, mask_stride_h, mask_stride_row};
  return run_fwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, scale, is_causal, dtype, stream,
                 BlockMask{nullptr, 0, 0, 0}, false, am, true);
}

extern "C" int sdpa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dO, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                               float scale, int is_causal, const void* attn_mask, long long mask_stride_b,
                               long long mask_stride_h, long long mask_stride_row, int dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
  const AddMask am{attn_mask, mask_stride_b, mask_stride_h, mask_stride_row};
  return run_bwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype,
                 workspace, workspace_bytes, stream, BlockMask{nullptr, 0, 0, 0}, false, am, true);
}

extern "C" int sdpa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int Lq, int Lk, int d, float scale, int is_causal, float dropout_p,
                                unsigned long long seed, int dtype, void* stream) {
  return run_fwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, scale, is_causal, dtype, stream,
                 BlockMask{nullptr, 0, 0, 0}, false, AddMask{nullptr, 0, 0, 0}, false, Dropout{dropout_p, seed});
}

extern "C" int sdpa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                                float scale, int is_causal, float dropout_p, unsigned long long seed, int dtype,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return run_bwd(self_shape(B, H, Lq, Lk, d, nullptr), q, k, v, o, lse, dO, dq, dk, dv, scale, is_causal, dtype,
                 workspace, workspace_bytes, stream, BlockMask{nullptr, 0, 0, 0}, false, AddMask{nullptr, 0, 0, 0},
                 false, Dropout{dropout_p, seed});
}

extern "C" int sdpa_device_status(void* stream, unsigned* bits) {
  g_last_error.clear();
  unsigned* ptr = nullptr;
  int rc = status_ptr(&ptr);
  if (rc != SDPA_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (word != 0) {
    e = cudaMemset(ptr, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  }
  if (bits) *bits = word;
  if (word & SDPA_STATUS_TIMEOUT) return fail(SDPA_ERR_TIMEOUT, "a kernel wait timed out (status 0x%x)", word);
  if (word & SDPA_STATUS_BOUNDS) return fail(SDPA_ERR_BOUNDS, "a device-side bounds check failed (status 0x%x)", word);
  if (word & SDPA_STATUS_SEQLEN) return fail(SDPA_ERR_ARG, "a packed sequence is longer than its bound or has queries but no keys (status 0x%x)", word);
  return SDPA_OK;
}

extern "C" int sdpa_trace_events(int which, void* begin_event, void* end_event) {
  g_last_error.clear();
  if (which != 0 && which != 1) return fail(SDPA_ERR_ARG, "trace target must be 0 (forward) or 1 (backward), got %d", which);
  if ((begin_event == nullptr) != (end_event == nullptr))
    return fail(SDPA_ERR_ARG, "trace events must both be set or both be NULL");
  g_trace_begin[which] = static_cast<cudaEvent_t>(begin_event);
  g_trace_end[which] = static_cast<cudaEvent_t>(end_event);
  return SDPA_OK;
}

extern "C" int sdpa_debug_set(int flags) {
  const int old = g_debug_flags;
  g_debug_flags = flags;
  return old;
}

extern "C" const char* sdpa_last_error(void) { return g_last_error.c_str(); }

extern "C" int sdpa_version(void) { return 100; }

extern "C" int sdpa_debug_build(void) {
#ifdef SDPA_DEBUG
  return 1;
#else
  return 0;
#endif
}
