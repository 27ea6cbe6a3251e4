// fwd_tc.cu -- exact attention forward on the sm_103a tensor cores.
//
// The IO-aware scheme of the FlashAttention news article (QbitAI repost,
// section "FlashAttention"): Q and K/V are tiled through shared memory so the
// Lq x Lk score matrix never reaches HBM, with the online-softmax rescale that
// keeps the tiled result exact and the per-row log-sum-exp saved for the
// backward. The article's loop order (K/V blocks outer, Q blocks inner, sized
// for an A100) is prior art; here each CTA owns 256 query rows (two 128-row
// tiles) of one (batch|sequence, head) and streams K/V blocks past them:
//
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into a ring of slots
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T and O_t += P_t V_j as
//               tcgen05.mma, accumulators in TMEM
//   warps 0-3   softmax for tile 0: one thread per query row reads its S row
//   warps 4-7   softmax for tile 1    from TMEM, masks, updates the running max
//               m and sum l, writes P (fp16/bf16) to shared memory, rescales
//               its O row in TMEM when m grew, and finally writes O = O/l and
//               LSE = (m + log2 l) ln 2.
//
// The two tiles alternate on the tensor cores: while one softmax group works
// on its tile, the MMAs of the other tile run. TMEM columns: S_0 [0,128),
// S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
#include <type_traits>

#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 128;          // keys per K/V block
constexpr int kThreads = 320;    // 8 softmax warps + producer + MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kBlk = D >= 64 ? 64 : D;             // elements per swizzled row
  static constexpr int kNBlk = D / kBlk;                      // column blocks per tile
  static constexpr uint32_t kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kRowBytes = kBlk * 2;                  // 128 or 64
  static constexpr int kSbo = 8 * kRowBytes;                  // 8-row group stride
  static constexpr int kColBlkBytes = 128 * kRowBytes;        // one column block of a 128-row tile
  static constexpr int kTileBytes = 128 * D * 2;              // a Q, K or V tile
  static constexpr int kPBytes = BM * BN * 2;                 // a P tile (two 64-key blocks)
  static constexpr int kSlots = D == 128 ? 3 : (D == 64 ? 6 : 8);
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = 2 * kTileBytes;
  static constexpr int kOffP = kOffSlots + kSlots * kTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kSmem = kOffBar + 512 + 1024;          // barriers + alignment slack
};

struct __align__(8) Bars {
  uint64_t q;
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t s[2];
  uint64_t p[2];
  uint64_t o[2];
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Number of K/V blocks tile rows [r, r+128) need.
template <bool CAUSAL>
__device__ __forceinline__ int tile_blocks(int r, int len_q, int len_k) {
  if (r >= len_q) return 0;
  const int nkv = (len_k + BN - 1) / BN;
  if (!CAUSAL) return nkv;
  const int last_row = min(r + BM - 1, len_q - 1);
  return min(nkv, last_row / BN + 1);
}

template <int D, typename T, bool CAUSAL, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const Problem p, const __grid_constant__ CUtensorMap tmQ,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);

  // ---- which unit and which rows
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int unit, pair, len_q, len_k, tok0 = 0, h = 0;
  {
    // Unit-major order: the CTAs of one (batch|sequence, head) run side by side
    // and share its K/V through L2; under causal masking the longest rows go first.
    const int npairs = ((PACKED ? p.Lk : p.Lq) + 2 * BM - 1) / (2 * BM);
    unit = blockIdx.x / npairs;
    const int ord = blockIdx.x % npairs;
    pair = CAUSAL ? (npairs - 1 - ord) : ord;
    if (PACKED) {
      const int s = unit / p.H;
      h = unit % p.H;
      tok0 = p.cu_seqlens[s];
      len_q = len_k = p.cu_seqlens[s + 1] - tok0;
      if (len_q > p.Lk && pair == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
    } else {
      len_q = p.Lq;
      len_k = p.Lk;
    }
  }
  const int r0 = pair * 2 * BM;
  const int n0 = tile_blocks<CAUSAL>(r0, len_q, len_k);
  const int n1 = tile_blocks<CAUSAL>(r0 + BM, len_q, len_k);
  const int nmax = max(n0, n1);
  if (nmax == 0) return;

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sSlots = smem_u32(smem + C::kOffSlots);
  const uint32_t sP = smem_u32(smem + C::kOffP);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s[t], 1);
      mbar_init(&bars->p[t], BM);
      mbar_init(&bars->o[t], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile uint32_t* abort_flag = &bars->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      auto c1 = [&](int row) { return PACKED ? h : row; };
      auto c2 = [&](int row) { return PACKED ? tok0 + row : unit; };
      if (!(p.debug & kDebugDropQArrive)) {
        const uint32_t qbytes = (n0 > 0 ? C::kTileBytes : 0) + (n1 > 0 ? C::kTileBytes : 0);
        mbar_expect_tx(&bars->q, qbytes);
        for (int t = 0; t < 2; ++t) {
          if ((t == 0 ? n0 : n1) == 0) continue;
          const int row = r0 + t * BM;
          for (int cb = 0; cb < C::kNBlk; ++cb)
            tma_load_3d(smem + C::kOffQ + t * C::kTileBytes + cb * C::kColBlkBytes, &tmQ, &bars->q,
                        cb * C::kBlk, c1(row), c2(row));
        }
      }
      int it = 0;
      for (int j = 0; j < nmax && !*abort_flag; ++j) {
        for (int kv = 0; kv < 2; ++kv, ++it) {
          const int slot = it % C::kSlots;
          const int round = it / C::kSlots;
          if (round > 0 && !mbar_wait(&bars->empty[slot], (round - 1) & 1, abort_flag, p.status)) break;
          mbar_expect_tx(&bars->full[slot], C::kTileBytes);
          const CUtensorMap* m = kv ? &tmV : &tmK;
          const int row = j * BN;
          for (int cb = 0; cb < C::kNBlk; ++cb)
            tma_load_3d(smem + C::kOffSlots + slot * C::kTileBytes + cb * C::kColBlkBytes, m, &bars->full[slot],
                        cb * C::kBlk, c1(row), c2(row));
        }
      }
      if (*abort_flag) {
        // Let copies already issued land before the CTA's shared memory is released.
        const int first = max(0, it - C::kSlots);
        for (int f = first; f < it; ++f) mbar_wait_drain(&bars->full[f % C::kSlots], (f / C::kSlots) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __half>::value ? 0u : 1u;
      constexpr uint32_t idS = idesc_f16(fmt, 0, 0, BM, BN);
      constexpr uint32_t idO = idesc_f16(fmt, 0, 1, BM, D);
      auto issue_qk = [&](int t, int slot) {
        const uint32_t qa = sQ + t * C::kTileBytes;
        const uint32_t kb = sSlots + slot * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks * 16 / C::kBlk) * C::kColBlkBytes + (ks * 16 % C::kBlk) * 2;
          mma_ss(tmem + t * BN, smem_desc(qa + off, 16, C::kSbo, C::kSw), smem_desc(kb + off, 16, C::kSbo, C::kSw),
                 idS, ks > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint32_t pa = sP + t * C::kPBytes;
        const uint32_t vb = sSlots + slot * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t a = smem_desc(pa + (ks / 4) * (BM * 128) + (ks % 4) * 32, 16, 1024, kSwizzle128B);
          const uint64_t b = smem_desc(vb + ks * 16 * C::kRowBytes, C::kColBlkBytes, C::kSbo, C::kSw);
          mma_ss(tmem + 2 * BN + t * D, a, b, idO, (acc || ks > 0) ? 1u : 0u);
        }
      };
      int it = 0;
      bool ok = mbar_wait(&bars->q, 0, abort_flag, p.status);
      if (ok) {
        const int slot = it % C::kSlots;
        ok = mbar_wait(&bars->full[slot], (it / C::kSlots) & 1, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          if (n0 > 0) { issue_qk(0, slot); mma_commit(&bars->s[0]); }
          if (n1 > 0) { issue_qk(1, slot); mma_commit(&bars->s[1]); }
          mma_commit(&bars->empty[slot]);
          ++it;
        }
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int vslot = it % C::kSlots;
        if (!(ok = mbar_wait(&bars->full[vslot], (it / C::kSlots) & 1, abort_flag, p.status))) break;
        ++it;
        const bool has_next = j + 1 < nmax;
        int kslot = 0;
        if (has_next) {
          kslot = it % C::kSlots;
          if (!(ok = mbar_wait(&bars->full[kslot], (it / C::kSlots) & 1, abort_flag, p.status))) break;
          ++it;
        }
        tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          const int nt = t == 0 ? n0 : n1;
          if (j >= nt) continue;
          if (!(ok = mbar_wait(&bars->p[t], j & 1, abort_flag, p.status))) break;
          tc_fence_after();
          issue_pv(t, vslot, j > 0);
          if (j == nt - 1) {
            mma_commit(&bars->o[t]);
          } else {
            issue_qk(t, kslot);
            mma_commit(&bars->s[t]);
          }
        }
        mma_commit(&bars->empty[vslot]);
        if (has_next) mma_commit(&bars->empty[kslot]);
      }
      mma_commit(&bars->done);
      mbar_wait_drain(&bars->done, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp / 4;
    const int nt = t == 0 ? n0 : n1;
    const int rt = r0 + t * BM;
    const int rl = threadIdx.x & 127;        // row within the tile == TMEM lane
    const int row = rt + rl;                  // row within the unit
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 2 * BN + t * D;
    const uint32_t pRow = sP + t * C::kPBytes + rl * 128;
    const float c = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // warp-uniform decision: the TMEM loads below are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s[t], j & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[BN];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_ld_wait();
      float* x = reinterpret_cast<float*>(sr);
      const int kbase = j * BN;
      const bool need_mask = (kbase + BN > len_k) || (CAUSAL && kbase + BN - 1 > rt);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int key = kbase + i;
          if (key >= len_k || (CAUSAL && key > row)) x[i] = -INFINITY;
        }
      }
      float mx = x[0];
#pragma unroll
      for (int i = 1; i < BN; ++i) mx = fmaxf(mx, x[i]);
      const float m_new = fmaxf(m, mx * c);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);
      float sum = 0.f;
#pragma unroll
      for (int chunk = 0; chunk < BN / 8; ++chunk) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = ex2_approx(fmaf(x[chunk * 8 + 2 * e], c, -m_use));
          const float b = ex2_approx(fmaf(x[chunk * 8 + 2 * e + 1], c, -m_use));
          sum += a + b;
          pk[e] = Pack2<T>::pack(a, b);
        }
        const uint32_t addr = pRow + (chunk / 8) * (BM * 128) + (((chunk % 8) ^ (rl & 7)) << 4);
        st_shared_v4(addr, pk[0], pk[1], pk[2], pk[3]);
      }
      l = l * alpha + sum;
      if (j > 0 && __any_sync(0xffffffffu, m_new > m)) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + cc * 32, o);
        }
        tmem_st_wait();
      }
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p[t]);
    }
    if (nt > 0 && ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o[t], 0, abort_flag, p.status));
    if (nt > 0 && ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool live = row < len_q;
      T* orow = static_cast<T*>(p.o) +
                (PACKED ? (static_cast<long long>(tok0 + row) * p.H + h) * D
                        : (static_cast<long long>(unit) * len_q + row) * D);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = Pack2<T>::pack(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            w.y = Pack2<T>::pack(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            w.z = Pack2<T>::pack(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            w.w = Pack2<T>::pack(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc * 32 + 8 * e) = w;
          }
        }
      }
      if (live) {
        const long long li = PACKED ? static_cast<long long>(h) * p.Lq + tok0 + row
                                    : static_cast<long long>(unit) * len_q + row;
        p.lse[li] = (m + __log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, typename T, bool CAUSAL, bool PACKED>
cudaError_t launch_one(const Problem& p, const FwdMaps& m, cudaStream_t s) {
  auto kern = fwd_tc_kernel<D, T, CAUSAL, PACKED>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  const int rows = PACKED ? p.Lk : p.Lq;
  const long long npairs = (rows + 2 * BM - 1) / (2 * BM);
  const long long units = static_cast<long long>(p.B) * p.H;
  const long long blocks = npairs * units;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(blocks), kThreads, Cfg<D>::kSmem, s>>>(p, m.q, m.k, m.v);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_d(const Problem& p, const FwdMaps& m, cudaStream_t s) {
  const bool packed = p.cu_seqlens != nullptr;
  if (p.causal) return packed ? launch_one<D, T, true, true>(p, m, s) : launch_one<D, T, true, false>(p, m, s);
  return packed ? launch_one<D, T, false, true>(p, m, s) : launch_one<D, T, false, false>(p, m, s);
}

}  // namespace

cudaError_t launch_fwd_tc(const Problem& p, int dtype, const FwdMaps& m, cudaStream_t s) {
  if (dtype == kF16) {
    if (p.d == 32) return launch_d<32, __half>(p, m, s);
    if (p.d == 64) return launch_d<64, __half>(p, m, s);
    if (p.d == 128) return launch_d<128, __half>(p, m, s);
  } else if (dtype == kBF16) {
    if (p.d == 32) return launch_d<32, __nv_bfloat16>(p, m, s);
    if (p.d == 64) return launch_d<64, __nv_bfloat16>(p, m, s);
    if (p.d == 128) return launch_d<128, __nv_bfloat16>(p, m, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
