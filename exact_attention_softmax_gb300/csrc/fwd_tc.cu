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
// on its tile, the MMAs of the other tile run. A softmax group releases S_t as
// soon as it holds the row in registers, so Q_t K_{j+1}^T runs under its
// exponentials; P is double-buffered in shared memory for d <= 64, and O is
// rescaled only when a row maximum grows past a threshold. TMEM columns:
// S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
#include <type_traits>

#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 128;          // keys per K/V block
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;      // first MMA warp (also allocates TMEM)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running maximum used in the exponent is only raised when a row's new
// maximum exceeds it by more than this (log2 units), so P <= 2^8 and O is
// rescaled rarely; the result is the same because O and l share the maximum.
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
  static constexpr int kBlk = D >= 64 ? 64 : D;             // elements per swizzled row
  static constexpr int kNBlk = D / kBlk;                      // column blocks per tile
  static constexpr uint32_t kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kRowBytes = kBlk * 2;                  // 128 or 64
  static constexpr int kSbo = 8 * kRowBytes;                  // 8-row group stride
  static constexpr int kColBlkBytes = 128 * kRowBytes;        // one column block of a 128-row tile
  static constexpr int kTileBytes = 128 * D * 2;              // a Q, K or V tile
  static constexpr int kSlots = D == 128 ? 5 : (D == 64 ? 12 : 16);
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = 2 * kTileBytes;
  static constexpr int kOffBar = kOffSlots + kSlots * kTileBytes;
  static constexpr int kSmem = kOffBar + 512 + 1024;          // barriers + alignment slack
  static_assert(kSmem <= 232448, "shared memory budget");
  // TMEM columns. P (BN fp16/bf16 per row, two per 32-bit column) has its own
  // columns when they fit; at d = 128 it overlays the upper half of S_t, which
  // is dead once the softmax group holds S_t in registers.
  static constexpr bool kPAlias = D == 128;
  static constexpr uint32_t kColS = 0;                        // + t * BN
  static constexpr uint32_t kColO = 2 * BN;                   // + t * D
  static constexpr uint32_t kColP = kPAlias ? BN / 2 : 2 * BN + 2 * D;   // + t * (kPAlias ? BN : BN / 2)
  static constexpr uint32_t kPStride = kPAlias ? BN : BN / 2;
  // MMA issue: with P in its own columns each Q tile gets its own MMA warp, so
  // the tiles' waits and issues do not serialise; when P overlays S the two
  // tiles' chains are serial and one warp alternating between them keeps the
  // tensor cores busier.
  static constexpr int kMmaWarps = kPAlias ? 1 : 2;
  static constexpr int kThreads = (8 + 1 + kMmaWarps) * 32;
  static_assert(kPAlias || kColP + 2 * (BN / 2) <= 512, "TMEM budget");
};

struct __align__(8) Bars {
  uint64_t q;
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t s_full[2];     // S_t written by the tensor cores
  uint64_t s_free[2];     // S_t read into registers by its softmax group
  uint64_t p_full[2];     // P_t in TMEM (and O_t rescaled)
  uint64_t pv_done[2];    // O_t += P_t V_j finished
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// (a0, a1) * (c, c) + (b, b) as one packed fp32x2 FMA.
__device__ __forceinline__ void fma2(float& o0, float& o1, float a0, float a1, float c, float b) {
  uint64_t x, y, z, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(c));
  asm("mov.b64 %0, {%1, %1};" : "=l"(z) : "f"(b));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(z));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o0), "=f"(o1) : "l"(r));
}
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  uint64_t x, y, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(a0), "f"(a1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(r));
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
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
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
      if (len_q > p.Lk && ord == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
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

  if (threadIdx.x == 0) {
    mbar_init(&bars->q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], C::kMmaWarps);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], BM);
      mbar_init(&bars->p_full[t], BM);
      mbar_init(&bars->pv_done[t], 1);
    }
    mbar_init(&bars->done, C::kMmaWarps);
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
  volatile uint32_t* abort_flag = &bars->abort_flag;
  // All 512 columns are allocated, so the allocation starts at lane 0, column
  // 0; the constant keeps TMEM addresses compile-time known. Anything else is
  // reported as a failed wait and the CTA drains.
  constexpr uint32_t tmem = 0;
  if (bars->tmem_base != 0u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1u;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      auto c1 = [&](int row) { return PACKED ? h : row; };
      auto c2 = [&](int row) { return PACKED ? tok0 + row : unit; };
      if (!(p.debug & kDebugDropQArrive) && !*abort_flag) {
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
      // ring order: K_0, V_0, K_1, V_1, ...
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
  } else if (warp >= kMmaWarp && warp < kMmaWarp + C::kMmaWarps) {
    // ------------------------------------------------------------ MMA issue
    // Warp w serves Q tiles [t_lo, t_hi); lane 0 issues. Every MMA warp
    // consumes every K/V fill: a slot's empty barrier takes one commit from each.
    const int t_lo = C::kMmaWarps == 2 ? warp - kMmaWarp : 0;
    const int t_hi = C::kMmaWarps == 2 ? t_lo + 1 : 2;
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __half>::value ? 0u : 1u;
      constexpr uint32_t idS = idesc_f16(fmt, 0, 0, BM, BN);
      constexpr uint32_t idO = idesc_f16(fmt, 0, 1, BM, D);
      // descriptors of the operand tiles; advancing the start address by `off`
      // bytes adds off >> 4 to the descriptor (the address field cannot carry)
      const uint64_t dQ = smem_desc(sQ, 16, C::kSbo, C::kSw);
      const uint64_t dSlot0K = smem_desc(sSlots, 16, C::kSbo, C::kSw);
      const uint64_t dSlot0V = smem_desc(sSlots, C::kColBlkBytes, C::kSbo, C::kSw);
      auto issue_qk = [&](int t, int slot) {
        const uint64_t a = dQ + ((t * C::kTileBytes) >> 4);
        const uint64_t b = dSlot0K + ((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks * 16 / C::kBlk) * C::kColBlkBytes + (ks * 16 % C::kBlk) * 2) >> 4;
          mma_ss(tmem + C::kColS + t * BN, a + off, b + off, idS, ks > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint64_t b = dSlot0V + ((slot * C::kTileBytes) >> 4);
        const uint32_t a = tmem + C::kColP + t * C::kPStride;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ts(tmem + C::kColO + t * D, a + ks * 8, b + ((ks * 16 * C::kRowBytes) >> 4), idO,
                 (acc || ks > 0) ? 1u : 0u);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort_flag, p.status); };
      auto full_wait = [&](int pos) { return wait(&bars->full[pos % C::kSlots], (pos / C::kSlots) & 1); };
      bool ok = wait(&bars->q, 0) && full_wait(0);
      if (ok) {
        tc_fence_after();
        for (int t = t_lo; t < t_hi; ++t) {
          if ((t == 0 ? n0 : n1) == 0) continue;
          issue_qk(t, 0);
          mma_commit(&bars->s_full[t]);
        }
        mma_commit(&bars->empty[0]);
      }
      for (int j = 0; j < nmax && ok; ++j) {
        // K_{j+1} sits at ring position 2j+2, V_j at 2j+1
        const bool has_next = j + 1 < nmax;
        const int kpos = 2 * j + 2, vpos = 2 * j + 1;
        if (has_next && !(ok = full_wait(kpos))) break;
        if (!(ok = full_wait(vpos))) break;
        tc_fence_after();
        for (int t = t_lo; t < t_hi && ok; ++t) {
          const int nt = t == 0 ? n0 : n1;
          if (j >= nt) continue;
          if (!C::kPAlias && j + 1 < nt) {
            // S_t may be overwritten once its softmax group holds it in registers
            if (!(ok = wait(&bars->s_free[t], j & 1))) break;
            tc_fence_after();
            issue_qk(t, kpos % C::kSlots);
            mma_commit(&bars->s_full[t]);
          }
          if (!(ok = wait(&bars->p_full[t], j & 1))) break;
          tc_fence_after();
          issue_pv(t, vpos % C::kSlots, j > 0);
          mma_commit(&bars->pv_done[t]);
          if (C::kPAlias && j + 1 < nt) {
            // P_t overlays S_t: the next S_t is issued behind the MMA that reads P_t
            issue_qk(t, kpos % C::kSlots);
            mma_commit(&bars->s_full[t]);
          }
        }
        mma_commit(&bars->empty[vpos % C::kSlots]);
        if (has_next) mma_commit(&bars->empty[kpos % C::kSlots]);
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
    const uint32_t tS = tmem + lane_off + C::kColS + t * BN;
    const uint32_t tO = tmem + lane_off + C::kColO + t * D;
    const uint32_t tP = tmem + lane_off + C::kColP + t * C::kPStride;
    const float c = p.scale * kLog2e;
    float m_run = -INFINITY, l = 0.f;        // maximum used in the exponent (base 2), running sum
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      // warp-uniform decision: the TMEM accesses that follow are warp-collective
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
    };
    for (int j = 0; j < nt; ++j) {
      if (!(ok = wait_all(&bars->s_full[t], j & 1))) break;
      tc_fence_after();
      uint32_t sr[BN];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_ld_wait();
      if (!C::kPAlias) {
        tc_fence_before();
        mbar_arrive(&bars->s_free[t]);
      }
      float* x = reinterpret_cast<float*>(sr);
      const int kbase = j * BN;
      if ((kbase + BN > len_k) || (CAUSAL && kbase + BN - 1 > rt)) {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int key = kbase + i;
          if (key >= len_k || (CAUSAL && key > row)) x[i] = -INFINITY;
        }
      }
      // row maximum: four independent chains of three-input max
      float mx0 = max3f(x[0], x[1], x[2]), mx1 = max3f(x[3], x[4], x[5]);
      float mx2 = max3f(x[6], x[7], x[8]), mx3 = max3f(x[9], x[10], x[11]);
#pragma unroll
      for (int i = 12; i < BN - 4; i += 8) {
        mx0 = max3f(mx0, x[i], x[i + 1]);
        mx1 = max3f(mx1, x[i + 2], x[i + 3]);
        mx2 = max3f(mx2, x[i + 4], x[i + 5]);
        mx3 = max3f(mx3, x[i + 6], x[i + 7]);
      }
      mx0 = max3f(mx0, x[BN - 4], x[BN - 3]);
      mx1 = max3f(mx1, x[BN - 2], x[BN - 1]);
      const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3)) * c;
      const bool grow = mx > m_run + kRescaleThreshold;
      const float m_new = grow ? mx : m_run;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);
      // exponentials into packed registers, stored to TMEM in two halves; the
      // first half is computed before waiting for P_t's columns to be free
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[BN / 4];
#pragma unroll
        for (int chunk = 0; chunk < BN / 16; ++chunk) {
          const float* xc = x + half * (BN / 2) + chunk * 8;
          float e[8];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            fma2(e[2 * u], e[2 * u + 1], xc[2 * u], xc[2 * u + 1], c, -m_use);
            e[2 * u] = ex2_approx(e[2 * u]);
            e[2 * u + 1] = ex2_approx(e[2 * u + 1]);
          }
          add2(s0, s1, e[0], e[1]);
          add2(s2, s3, e[2], e[3]);
          add2(s0, s1, e[4], e[5]);
          add2(s2, s3, e[6], e[7]);
#pragma unroll
          for (int u = 0; u < 4; ++u) pk[chunk * 4 + u] = Pack2<T>::pack(e[2 * u], e[2 * u + 1]);
        }
        // P_t's columns are free once O_t += P_{j-1} V_{j-1} has finished (at d = 128
        // they overlay S_t, already in registers, and that MMA finished before S_j)
        if (half == 0 && !C::kPAlias && j > 0) ok = wait_all(&bars->pv_done[t], (j - 1) & 1);
        if (!ok) break;
        tmem_st32(tP + half * 32, pk);
      }
      if (!ok) break;
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      m_run = m_new;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O_t holds P_{j-1} V_{j-1} here: waited above, or (d = 128) finished before S_j
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 16; ++cc) {
          uint32_t o[16];
          tmem_ld16(tO + cc * 16, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(tO + cc * 16, o);
        }
        tmem_st_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
    }
    if (nt > 0 && ok) ok = wait_all(&bars->pv_done[t], (nt - 1) & 1);
    if (nt > 0 && ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool live = row < len_q;
      T* orow = static_cast<T*>(p.o) +
                (PACKED ? (static_cast<long long>(tok0 + row) * p.H + h) * D
                        : (static_cast<long long>(unit) * len_q + row) * D);
#pragma unroll 1
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
        p.lse[li] = (m_run + __log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
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
  kern<<<static_cast<unsigned>(blocks), Cfg<D>::kThreads, Cfg<D>::kSmem, s>>>(p, m.q, m.k, m.v);
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
