// bwd_persist.cu -- the tensor-core backward for d <= 64 on dense batches of
// plain or strided tensors, as persistent CTAs.
//
// The steps are those of bwd_tc.cu (same warp roles, TMEM plan and handoffs,
// described there). Here each CTA, one per SM, claims 128-key blocks of any
// unit from a dynamic queue and runs them one after another:
//   - the producer claims the next block (an atomic counter, one slot per
//     launch) and publishes it through a two-entry queue in shared memory to
//     the MMA, dQ-drain and softmax warps;
//   - K/V are double-buffered, so the next block's keys load while the
//     current block's query steps run; a buffer is reloaded once the MMAs of
//     the block that used it have read it (kv_empty);
//   - barrier phases run on a global step count across blocks;
//   - a block's dK / dV are read out of TMEM, then staged through the dS^T
//     buffer (the Q/dO stages already hold the next block's rows) and stored,
//     while the next block's S^T / dP^T MMAs run; its first dV / dK MMAs wait
//     for that read-out (acc_free).
// So the K/V load and the tail of one key block overlap the next block's
// work, where one CTA per key block (bwd_tc.cu) pays them in turn: the causal
// 32 x 8 x 1024 x 64 backward measured 3 % faster. d = 128 has no room for a
// second K/V buffer and stays in bwd_tc.cu, as do the block-sparse, mask and
// dropout kernels and packed batches: with a few query steps per key block,
// one CTA per key block measured faster on those (the 32-sequence causal
// packed backward 70 against 78 us, the packed cross-attention one 97 against
// 105 us, even with the empty key blocks past a sequence's end kept off the
// queue). The template keeps its packed form (PACKED), which passed the
// packed parity tests, but the dispatcher below does not launch it.
#include <algorithm>
#include <atomic>

#include "bwd_common.cuh"

namespace sdpa {
namespace {

constexpr int kPBarBytes = 320;    // shared memory for the barrier block
constexpr int kBSchedSlots = 1024;
__device__ unsigned g_bwd_sched[2 * kBSchedSlots];   // work counters (one pair per launch slot)

// The shared memory map of bwd_tc.cu with K/V double-buffered (and no mask or
// block list region).
template <int D, int EXT>
struct PCfg : BCfg<D, EXT> {
  using B = BCfg<D, EXT>;
  static constexpr int kKVBufs = 2;
  static constexpr int kOffK = 0;                                          // K of buffer b at + 2 b kKTile
  static constexpr int kOffV = kOffK + B::kKTile;                          // V likewise
  static constexpr int kOffQ = kKVBufs * 2 * B::kKTile;                    // kStages Q tiles
  static constexpr int kOffDO = kOffQ + B::kStages * B::kQTile;            // kStages dO tiles
  static constexpr int kOffDST = kOffDO + B::kStages * B::kQTile;          // dS^T, then the dK / dV staging
  static constexpr int kOffDQ = kOffDST + B::kPBytes;
  static constexpr int kOffStat = kOffDQ + B::kDqBytes;                    // kStages x (lse2[BQ], delta[BQ])
  static constexpr int kOffDqStage = kOffStat + B::kStages * B::BQ * 8;
  static constexpr int kOffBar = kOffDqStage + B::kDqStageBytes;
  static constexpr int kSmem = kOffBar + kPBarBytes + 1024;
  static_assert(D <= 64 && !B::kDqT, "d <= 64: dQ with the query rows on TMEM lanes");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct __align__(8) PBars {
  uint64_t kv[2];         // K/V buffer b loaded
  uint64_t kv_empty[2];   // the MMAs of the key block in buffer b that read K/V finished
  uint64_t acc_free;      // the last key block's dV / dK read out of TMEM
  uint64_t item_full[2];  // work-item queue from the producer to the other roles
  uint64_t item_empty[2];
  int item[2];
  uint64_t full[3];
  uint64_t empty[3];
  uint64_t s_full;        // S^T of the current step in TMEM
  uint64_t dp_full;       // dP^T of the current step in TMEM
  uint64_t s_free;        // S^T and dP^T read into registers by both softmax groups
  uint64_t pds_full;      // P^T in TMEM, dS^T in shared memory
  uint64_t pds_free;      // ... consumed by the dV, dK, dQ MMAs
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t kv_done;       // a key block's dV / dK MMAs finished
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(PBars) <= kPBarBytes, "the barrier block's shared memory");

// Packed fp32x2 arithmetic (one instruction for two lanes of values):
// (a0, a1) * (c, c) + (b0, b1), (a0, a1) - (b0, b1) and (a0, a1) * (b0, b1).
__device__ __forceinline__ uint64_t pack_f32x2(float a0, float a1) {
  uint64_t x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  return x;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t x, float& a0, float& a1) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(x));
}
__device__ __forceinline__ void fma2v(float& o0, float& o1, float a0, float a1, float c, float b0, float b1) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pack_f32x2(a0, a1)), "l"(pack_f32x2(c, c)), "l"(pack_f32x2(b0, b1)));
  unpack_f32x2(r, o0, o1);
}
__device__ __forceinline__ void sub2(float& o0, float& o1, float a0, float a1, float b0, float b1) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pack_f32x2(a0, a1)), "l"(pack_f32x2(b0, b1)));
  unpack_f32x2(r, o0, o1);
}
__device__ __forceinline__ void mul2(float& o0, float& o1, float a0, float a1, float b0, float b1) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pack_f32x2(a0, a1)), "l"(pack_f32x2(b0, b1)));
  unpack_f32x2(r, o0, o1);
}

template <int D, typename T, bool CAUSAL, bool PACKED, int EXT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_persist_kernel(const BwdProblem bp, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              unsigned* sched) {
  using C = PCfg<D, EXT>;
  // plain (EXT 0) or strided (EXT 4) tensors
  constexpr bool STRIDED = EXT == 4;
  static_assert(EXT == 0 || EXT == 4, "plain or strided tensors");
  constexpr int BQ = C::BQ;
  constexpr int NH = C::kHalf;     // query columns per softmax group, taken in one piece
  const Problem& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PBars* bars = reinterpret_cast<PBars*>(smem + C::kOffBar);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Packed batches: a unit is (sequence, head); its queries are rows
  // cu_seqlens[s] .. cu_seqlens[s+1]-1 of the query token axis, its keys rows
  // cu_k[s] .. cu_k[s+1]-1 of the key token axis, and p.Lk bounds every key length.
  const int nkb = (p.Lk + BK - 1) / BK;
  const int nitems = nkb * p.B * p.H;
  // A work item is one 128-key block of one unit. Items go out in groups of
  // bp.group units; inside a group key block 0 of every unit comes first,
  // then key block 1, and so on. Under causal masking low key blocks see the
  // most query rows, so the longest items start first, while a group's Q, dO
  // and dQ accumulator stay small enough for L2.
  struct Item {
    int unit, kblk, key0, Lq, Lk, tok0, tok0k, head, nq, i0;
    long long row0, row0k, stat0;
    bool bad;       // packed: lengths outside their bounds (reported, nothing written)
    bool valid;     // lengths within bounds and the key block inside the unit
  };
  auto decode = [&](int idx) {
    Item x;
    const int per_group = bp.group * nkb;
    const int grp = idx / per_group, rg = idx % per_group;
    const int gunits = min(bp.group, p.B * p.H - grp * bp.group);
    x.unit = grp * bp.group + rg % gunits;
    x.kblk = rg / gunits;
    x.key0 = x.kblk * BK;
    x.Lq = p.Lq;
    x.Lk = p.Lk;
    x.tok0 = x.tok0k = x.head = 0;
    x.bad = false;
    if (PACKED) {
      const int sq = x.unit / p.H;
      x.head = x.unit % p.H;
      x.tok0 = p.cu_seqlens[sq];
      x.Lq = p.cu_seqlens[sq + 1] - x.tok0;
      x.tok0k = p.cu_k[sq];
      x.Lk = p.cu_k[sq + 1] - x.tok0k;
      x.bad = x.Lq > p.max_q || x.Lk > p.Lk || (x.Lq > 0 && x.Lk <= 0);
    }
    x.valid = !x.bad && x.key0 < x.Lk;
    // element offset of row 0 of this unit (query side, key side) and of its
    // row statistics (dense: [B,H,L,d] and [B,H,L]; packed: [total,H,d] and [H,total])
    x.row0 = PACKED ? (static_cast<long long>(x.tok0) * p.H + x.head) * D : 0;
    x.row0k = PACKED ? (static_cast<long long>(x.tok0k) * p.H + x.head) * D : 0;
    x.stat0 = PACKED ? static_cast<long long>(x.head) * p.Lq + x.tok0 : static_cast<long long>(x.unit) * x.Lq;
    x.nq = (x.Lq + BQ - 1) / BQ;
    x.i0 = CAUSAL ? min(x.nq, x.key0 / BQ) : 0;
    return x;
  };
  // rows of a unit are rstride elements apart
  const long long rstride = PACKED ? static_cast<long long>(p.H) * D : D;
  // K / V of buffer b
  auto sK = [&](int b) { return smem_u32(smem + C::kOffK + b * 2 * C::kKTile); };
  auto sV = [&](int b) { return smem_u32(smem + C::kOffV + b * 2 * C::kKTile); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sDST = smem_u32(smem + C::kOffDST);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);   // [stage][2][BQ]

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kv[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->item_full[i], 1);
      mbar_init(&bars->item_empty[i], 14);   // S, G, 4 dQ drain and 8 softmax warps
    }
    mbar_init(&bars->acc_free, 256);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->full[i], 32);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->dq_full[i], 1);
      mbar_init(&bars->dq_free[i], 128);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->s_free, 256);
    mbar_init(&bars->pds_full, 256);
    mbar_init(&bars->pds_free, 2);     // dV/dK warp and dQ warp
    mbar_init(&bars->kv_done, 1);
    mbar_init(&bars->done, 2);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaSWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile uint32_t* abort_flag = &bars->abort_flag;
  // query steps of an item, and the query step (in BQ rows) of its st-th step
  // (from the item's scalars, so that no Item is kept across a step loop)
  auto nsteps_of = [&](const Item& x) { return x.nq - x.i0; };
  auto qstep_at = [&](int i0, int nq, int st) { return i0 + st; };
  // The roles walk the CTA's items from the producer's queue (entry kk % 2;
  // -1 ends it).
  auto take = [&](int kk, int& idx) {
    if (!mbar_wait(&bars->item_full[kk & 1], (kk >> 1) & 1, abort_flag, p.status)) return false;
    idx = *reinterpret_cast<volatile int*>(&bars->item[kk & 1]);
    return true;
  };
  // ... and hand the queue entry back: one arrival per consuming warp, from
  // its lane 0 once every lane has read it (lane_only: roles run by lane 0)
  auto give_back = [&](int kk, bool lane_only) {
    if (!lane_only) __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bars->item_empty[kk & 1]);
  };
  // All 512 columns are allocated, so the allocation starts at column 0.
  constexpr uint32_t tmem = 0;
  if (bars->tmem_base != 0u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1u;
  }

  if (warp >= kDqWarp0) {
   regs_dec<kRegsOther>();
   if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    int kv = 0;              // items run so far (K/V buffer kv % kKVBufs, its phases)
    int g0 = 0;              // steps of those items (the Q/dO stages' phases)
    int claim = blockIdx.x;  // persistent: the next item to publish
    bool ok = true;
    for (int kk = 0; ok; ++kk) {
      int idx = -1;
      {
        // publish the next item (or the end marker) on the queue, then claim the one after it
        int pub = -2;
        if (lane == 0) {
          const int cur = claim < nitems ? claim : -1;
          const int q = kk & 1;
          if (kk < 2 || mbar_wait(&bars->item_empty[q], ((kk >> 1) - 1) & 1, abort_flag, p.status)) {
            bars->item[q] = cur;
            mbar_arrive(&bars->item_full[q]);
            pub = cur;
            if (cur >= 0) claim = static_cast<int>(atomicAdd(sched, 1u)) + static_cast<int>(gridDim.x);
          }
        }
        idx = __shfl_sync(0xffffffffu, pub, 0);
        if (idx == -2) ok = false;
        if (idx < 0) break;
      }
      const Item x = decode(idx);
      if (x.bad && x.kblk == 0 && lane == 0) atomicOr(p.status, kStatusSeqlen);
      if (!x.valid) continue;
      const int nsteps = nsteps_of(x);
      const int unit = x.unit, head = x.head, Lq = x.Lq, tok0 = x.tok0, i0 = x.i0, nq = x.nq;
      // boxes: packed (column, head, token); dense (column, row, unit), or
      // (column, row, head, batch) through 4-D maps of strided tensors
      auto load = [&](void* dst, const CUtensorMap* m, uint64_t* bar, int col, int row, int tok) {
        if constexpr (PACKED) tma_load_3d(dst, m, bar, col, head, tok + row);
        else if constexpr (STRIDED) tma_load_4d(dst, m, bar, col, row, unit % p.H, unit / p.H);
        else tma_load_3d(dst, m, bar, col, row, unit);
      };
      // K / V into buffer b once the MMAs of the item that used it last have read it
      const int b = kv % C::kKVBufs;
      ok = !*abort_flag;
      if (lane == 0 && ok) {
        if (kv >= C::kKVBufs)
          ok = mbar_wait(&bars->kv_empty[b], ((kv / C::kKVBufs) - 1) & 1, abort_flag, p.status);
        if (ok) {
          mbar_expect_tx(&bars->kv[b], 2 * C::kKTile);
          for (int cb = 0; cb < C::kNBlk; ++cb) {
            load(smem + C::kOffK + b * 2 * C::kKTile + cb * C::kKColBlk, &tmK, &bars->kv[b], cb * C::kBlk, x.key0,
                 x.tok0k);
            load(smem + C::kOffV + b * 2 * C::kKTile + cb * C::kKColBlk, &tmV, &bars->kv[b], cb * C::kBlk, x.key0,
                 x.tok0k);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      ++kv;
      const float* lse = p.lse + x.stat0;
      const float* delta = bp.delta + x.stat0;
      // The row statistics of step s + 1 are fetched into registers while step s
      // is in flight, so their latency hides behind the wait for a free stage.
      constexpr int kPer = BQ / 32;
      float nl[kPer], nd[kPer];
      auto fetch = [&](int step) {
        const int q0 = qstep_at(i0, nq, step) * BQ;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int q = q0 + lane + 32 * u;
          const bool in = step < nsteps && q < Lq;
          // a row with no visible key (LSE = -inf) gets +inf, so all its P are 0
          const float lq = in ? lse[q] : INFINITY;
          nl[u] = lq == -INFINITY ? INFINITY : lq * kLog2e;
          nd[u] = in ? delta[q] : 0.f;
        }
      };
      fetch(0);
      int s = 0;
      for (; s < nsteps; ++s) {
        const int g = g0 + s;   // global step
        const int stage = g % C::kStages, round = g / C::kStages;
        ok = !*abort_flag;
        if (ok && lane == 0 && round > 0) ok = mbar_wait(&bars->empty[stage], (round - 1) & 1, abort_flag, p.status);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const int q0 = qstep_at(i0, nq, s) * BQ;
        if (lane == 0) {
          mbar_expect_tx_only(&bars->full[stage], 2 * C::kQTile);
          for (int cb = 0; cb < C::kNBlk; ++cb) {
            load(smem + C::kOffQ + stage * C::kQTile + cb * C::kQColBlk, &tmQ, &bars->full[stage], cb * C::kBlk, q0,
                 tok0);
            load(smem + C::kOffDO + stage * C::kQTile + cb * C::kQColBlk, &tmDO, &bars->full[stage], cb * C::kBlk, q0,
                 tok0);
          }
        }
        float* st = stat + stage * 2 * BQ;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          st[lane + 32 * u] = nl[u];
          st[BQ + lane + 32 * u] = nd[u];
        }
        mbar_arrive(&bars->full[stage]);
        fetch(s + 1);
      }
      g0 += s;
    }
    // the last claimer to finish resets this launch's scheduler slot
    if (lane == 0 && atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(sched, 0u);
      atomicExch(sched + 1, 0u);
    }
    if (lane == 0 && *abort_flag) {
      // let copies already issued land before the CTA's shared memory is released
      for (int k = max(0, kv - C::kKVBufs); k < kv; ++k) mbar_wait_drain(&bars->kv[k % C::kKVBufs], (k / C::kKVBufs) & 1);
      for (int f = max(0, g0 - C::kStages); f < g0; ++f)
        mbar_wait_drain(&bars->full[f % C::kStages], (f / C::kStages) & 1);
    }
   } else if (warp == kMmaSWarp || warp == kMmaGWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __half>::value ? 0u : 1u;
      auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort_flag, p.status); };
      bool ok = true;
      // dQ partial of global step t (K of buffer b): contraction over the 128
      // keys, both operands MN-major
      constexpr uint32_t idQ = idesc_f16(fmt, 1, 1, BQ, D);   // dQ: M = queries, N = D
      const uint64_t dDSm = smem_desc(sDST, C::kPColBlk, 1024, kSwizzle128B);
      auto issue_dq = [&](int t, int b) {
        if (!wait(&bars->pds_full, t & 1)) return false;
        const int buf = 0;
        if (t >= 1 && !wait(&bars->dq_free[0], (t - 1) & 1)) return false;
        tc_fence_after();
        const uint64_t dKm = smem_desc(sK(b), C::kKColBlk, C::kSbo, C::kSw);
        const uint32_t tdq = tmem + C::kTdQ + buf * C::kDqCols;
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint32_t kb_off = (ks * 16 * C::kRowBytes) >> 4;   // 16 key rows of the K tile
          const uint32_t ds_off = (ks * 16 * 128) >> 4;            // 16 key rows of dS^T
          mma_ss(tdq, dDSm + ds_off, dKm + kb_off, idQ, ks > 0);
        }
        mma_commit(&bars->dq_full[buf]);
        mma_commit(&bars->pds_free);
        return true;
      };
      int kv = 0;              // items run so far (K/V buffer kv % kKVBufs)
      int g0 = 0;              // their steps (the global step index of this item's first)
      for (int kk = 0; ok; ++kk) {
        int idx;
        if (!(ok = take(kk, idx))) break;
        give_back(kk, true);
        if (idx < 0) break;
        const Item x = decode(idx);
        if (!x.valid) continue;
        const int nsteps = nsteps_of(x);
        const int b = kv % C::kKVBufs;
        if (warp == kMmaSWarp) {
          // S^T = K Q^T and dP^T = V dO^T (K-major operands, contraction over D),
          // and the dQ partial of the previous step
          constexpr uint32_t idS = idesc_f16(fmt, 0, 0, BK, BQ);
          if (!(ok = wait(&bars->kv[b], (kv / C::kKVBufs) & 1))) break;
          const uint64_t dK0 = smem_desc(sK(b), 16, C::kSbo, C::kSw);
          const uint64_t dV0 = smem_desc(sV(b), 16, C::kSbo, C::kSw);
          const uint64_t dQ0 = smem_desc(sQ, 16, C::kSbo, C::kSw);
          const uint64_t dO0 = smem_desc(sDO, 16, C::kSbo, C::kSw);
          for (int s = 0; s < nsteps && ok; ++s) {
            const int g = g0 + s;   // global step
            const int stage = g % C::kStages;
            if (!(ok = wait(&bars->full[stage], (g / C::kStages) & 1))) break;
            if (g > 0 && !(ok = wait(&bars->s_free, (g - 1) & 1))) break;
            tc_fence_after();
            const uint32_t qoff = (stage * C::kQTile) >> 4;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t cb = ks * 16 / C::kBlk, within = (ks * 16 % C::kBlk) * 2;
              const uint32_t ko = (cb * C::kKColBlk + within) >> 4, qo = qoff + ((cb * C::kQColBlk + within) >> 4);
              mma_ss(tmem + C::kTS, dK0 + ko, dQ0 + qo, idS, ks > 0);
            }
            // S^T alone lets the softmax groups start on P while dP^T computes
            mma_commit(&bars->s_full);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t cb = ks * 16 / C::kBlk, within = (ks * 16 % C::kBlk) * 2;
              const uint32_t ko = (cb * C::kKColBlk + within) >> 4, qo = qoff + ((cb * C::kQColBlk + within) >> 4);
              mma_ss(tmem + C::kTdP, dV0 + ko, dO0 + qo, idS, ks > 0);
            }
            mma_commit(&bars->dp_full);
            // dQ of this item's previous step: needs its dS^T and a free dQ buffer
            if (s > 0 && !(ok = issue_dq(g - 1, b))) break;
          }
          if (ok && nsteps > 0) ok = issue_dq(g0 + nsteps - 1, b);
          // every MMA of this item that reads K/V has been issued: the buffer may be reloaded after them
          mma_commit(&bars->kv_empty[b]);
        } else {
          // dV += P^T dO, dK += dS^T Q (A K-major over queries, B MN-major)
          constexpr uint32_t idKV = idesc_f16(fmt, 0, 1, BK, D);
          const uint64_t dDST = smem_desc(sDST, 16, 1024, kSwizzle128B);
          const uint64_t dQm = smem_desc(sQ, C::kQColBlk, C::kSbo, C::kSw);
          const uint64_t dOm = smem_desc(sDO, C::kQColBlk, C::kSbo, C::kSw);
          for (int s = 0; s < nsteps && ok; ++s) {
            const int g = g0 + s;   // global step
            const int stage = g % C::kStages;
            const uint32_t qoff = (stage * C::kQTile) >> 4;
            // the item's first dV / dK overwrite the accumulators: the last
            // item's epilogue must have read them
            if (s == 0 && kv > 0 && !(ok = wait(&bars->acc_free, (kv - 1) & 1))) break;
            if (!(ok = wait(&bars->pds_full, g & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks) {
              const uint32_t aoff = ((ks / 4) * C::kPColBlk + (ks % 4) * 32) >> 4;
              const uint32_t boff = qoff + ((ks * 16 * C::kRowBytes) >> 4);
              const uint32_t acc = (s > 0 || ks > 0) ? 1u : 0u;
              mma_ts(tmem + C::kTdV, tmem + C::kTP + ks * 8, dOm + boff, idKV, acc);
              mma_ss(tmem + C::kTdK, dDST + aoff, dQm + boff, idKV, acc);
            }
            mma_commit(&bars->pds_free);
            mma_commit(&bars->empty[stage]);
          }
          // this item's dV / dK are complete once its MMAs are
          mma_commit(&bars->kv_done);
        }
        g0 += nsteps;
        ++kv;
      }
      mma_commit(&bars->done);
      mbar_wait_drain(&bars->done, 0);
    }
   } else if (warp < kDqWarp0 + 4) {
    // ------------------------------------------------ dQ drain
    // lane = query row: 16-byte vector reductions of whole row segments (as
    // in bwd_tc.cu at d <= 64)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const long long dq_ext = bp.acc_rows * D;   // elements of the accumulator (debug bounds checks)
    int g0 = 0;                                  // global step index of the item's first step
    bool ok = true;
    for (int kk = 0; ok; ++kk) {
     int idx;
     ok = __all_sync(0xffffffffu, take(kk, idx));
     if (!ok) break;
     give_back(kk, false);
     if (idx < 0) break;
     const Item x = decode(idx);
     if (!x.valid) continue;
     const int nsteps = nsteps_of(x);
     const int Lq = x.Lq, i0 = x.i0, nq = x.nq;
     const long long dq_base = PACKED ? x.row0 : static_cast<long long>(x.unit) * Lq * D;
     float* dq_unit = bp.dq_acc + dq_base;
     for (int s = 0; s < nsteps; ++s) {
      const int g = g0 + s;   // global step
      const int buf = 0;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->dq_full[0], g & 1, abort_flag, p.status)))) break;
      tc_fence_after();
      const int q0 = qstep_at(i0, nq, s) * BQ;
      const uint32_t tdq = tmem + lane_off + C::kTdQ + buf * C::kDqCols;
      // lane = query row: each 32-column piece of the warp's 32 rows goes
      // through its 4 KB staging area (16-byte chunk c of row i at slot
      // c ^ (i % 8)) and out as 16-byte reductions that cover four whole
      // 128-byte row segments per instruction, not 32 scattered rows
      const int lane = threadIdx.x & 31;
      const int rbase = q0 + (warp & 3) * 32;                  // query row of lane 0
      const uint32_t stg = smem_u32(smem + C::kOffDqStage + (warp - kDqWarp0) * 4096);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tdq + cc * 32, o);
        tmem_ld_wait();
        if (cc == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&bars->dq_free[buf]);
        }
        __syncwarp();                                          // the previous piece has been read
#pragma unroll
        for (int e = 0; e < 8; ++e)
          st_shared_v4(stg + (lane * 8 + (e ^ (lane & 7))) * 16, o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        __syncwarp();
        const int c = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + lane / 8;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(stg + (rr * 8 + (c ^ (rr & 7))) * 16) : "memory");
          const long long qo = static_cast<long long>(rbase + rr) * rstride + cc * 32 + c * 4;
          if (rbase + rr < Lq && SDPA_CHECK(dq_base + qo + 4 <= dq_ext, p.status))
            red_add_v4_f32(dq_unit + qo, w0, w1, w2, w3);
        }
      }
     }
     g0 += nsteps;
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------ P^T and dS^T, then dV / dK
    const int half = warp / 4;                                // query columns [half * kHalf, +kHalf)
    const int r = threadIdx.x & 127;                          // key row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale * kLog2e;
    bool ok = true;
    int kv = 0;              // items run so far (the phases of kv_done / acc_free)
    int g0 = 0;              // their steps (the global step index of this item's first)
    for (int kk = 0; ok; ++kk) {
     int idx;
     ok = __all_sync(0xffffffffu, take(kk, idx));
     if (!ok) break;
     give_back(kk, false);
     if (idx < 0) break;
     const Item x = decode(idx);
     if (!x.valid) continue;
     const int nsteps = nsteps_of(x);
     const int key0 = x.key0, Lk = x.Lk, unit = x.unit, i0 = x.i0;
     const long long row0k = x.row0k;
     const int key = key0 + r;
     for (int s = 0; s < nsteps; ++s) {
      const int g = g0 + s;   // global step
      const int stage = g % C::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, g & 1, abort_flag, p.status) &&
                                       mbar_wait(&bars->full[stage], (g / C::kStages) & 1, abort_flag, p.status) &&
                                       mbar_wait(&bars->dp_full, g & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[NH], dv[NH];
#pragma unroll
      for (int cc = 0; cc < NH / 32; ++cc) {
        tmem_ld32(tmem + lane_off + C::kTS + half * NH + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[cc * 32]));
        tmem_ld32(tmem + lane_off + C::kTdP + half * NH + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[cc * 32]));
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->s_free);               // the next S^T / dP^T may be written
      const int q0 = (i0 + s) * BQ + half * NH;  // this group's first query column
      const bool need_mask = (CAUSAL && q0 < key0 + BK - 1) || (key0 + BK > Lk);
      // row statistics of these query columns (written by the producer
      // before it arrived on full[stage])
      const float* slf = stat + stage * 2 * BQ + half * NH;
      uint32_t pk[NH / 2], dk[NH / 2];
      // P = 2^(S * scale * log2(e) - LSE2), dS = P * (dP - D), packed; the
      // per-element causal / length test only where the tile needs it
      auto body = [&](auto masked) {
        constexpr bool M = decltype(masked)::value;
#pragma unroll
        for (int gq = 0; gq < NH / 4; ++gq) {
          float l4[4], d4[4];
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(l4[0]), "=f"(l4[1]), "=f"(l4[2]), "=f"(l4[3]) : "r"(smem_u32(slf + 4 * gq)));
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(d4[0]), "=f"(d4[1]), "=f"(d4[2]), "=f"(d4[3]) : "r"(smem_u32(slf + BQ + 4 * gq)));
          float pr[4], ds[4];
#pragma unroll
          for (int h = 0; h < 4; h += 2) {
            // two columns per packed fp32x2 instruction
            const int col = 4 * gq + h;
            float e0, e1, t0, t1;
            fma2v(e0, e1, __uint_as_float(sv[col]), __uint_as_float(sv[col + 1]), c, -l4[h], -l4[h + 1]);
            float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
            if (M && ((CAUSAL && q0 + col < key) || key >= Lk)) p0 = 0.f;
            if (M && ((CAUSAL && q0 + col + 1 < key) || key >= Lk)) p1 = 0.f;
            sub2(t0, t1, __uint_as_float(dv[col]), __uint_as_float(dv[col + 1]), d4[h], d4[h + 1]);
            mul2(ds[h], ds[h + 1], p0, p1, t0, t1);
            pr[h] = p0;
            pr[h + 1] = p1;
          }
          pk[2 * gq] = Pack2<T>::pack(pr[0], pr[1]);
          pk[2 * gq + 1] = Pack2<T>::pack(pr[2], pr[3]);
          dk[2 * gq] = Pack2<T>::pack(ds[0], ds[1]);
          dk[2 * gq + 1] = Pack2<T>::pack(ds[2], ds[3]);
        }
      };
      if (need_mask) body(std::true_type{});
      else body(std::false_type{});
      // P^T / dS^T buffers are free once the previous step's dV, dK, dQ MMAs finished
      if (g > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->pds_free, (g - 1) & 1, abort_flag, p.status));
      if (!ok) break;
      // P^T into TMEM (this thread's key row, two queries per column), dS^T
      // into shared memory: [key row][query] in 128-byte swizzled rows, 64
      // queries per column block
      tmem_st32(tmem + lane_off + C::kTP + (half * NH) / 2, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
#pragma unroll
      for (int c8 = 0; c8 < NH / 8; ++c8) {
        const int chunk = half * (NH / 8) + c8;   // 8-query chunk index within the tile
        const uint32_t off = (chunk / 8) * C::kPColBlk + r * 128 + (((chunk % 8) ^ (r & 7)) << 4);
        st_shared_v4(sDST + off, dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2], dk[4 * c8 + 3]);
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bars->pds_full);
     }
     if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_done, kv & 1, abort_flag, p.status));
     // persistent: the staging below reuses the dS^T buffer, which the item's
     // last dK and dQ MMAs read
     if (ok && nsteps > 0)
       ok = __all_sync(0xffffffffu, mbar_wait(&bars->pds_free, (g0 + nsteps - 1) & 1, abort_flag, p.status));
     if (ok) {
      // group 0 writes dV, group 1 writes dK = scale * dK_acc. Every MMA of
      // the item has finished (kv_done), so each warp stages its 32 rows in
      // shared memory: the Q/dO stages (one item per CTA), or in a persistent
      // kernel, whose next item's Q/dO are already loading, the dS^T buffer's
      // part this warp alone writes (16-byte chunk c of row r at slot
      // c ^ f(r), f(r) = r % 8, or (r / 2) % 4 for the 4-chunk rows of d = 32:
      // the 8 lanes of a quarter-warp hit 8 different bank groups), and stores
      // them back whole rows per instruction instead of 32 rows of 16 bytes.
      tc_fence_after();
      const uint32_t col0 = half == 0 ? C::kTdV : C::kTdK;
      const float sc = half == 0 ? 1.f : p.scale;
      const long long out_off = PACKED    ? row0k + static_cast<long long>(key) * rstride
                                : STRIDED ? dense_off(p, half == 0 ? kTdv : kTdk, unit / p.H, unit % p.H, key)
                                          : (static_cast<long long>(unit) * Lk + key) * D;
      T* out = static_cast<T*>(half == 0 ? bp.dv : bp.dk) + out_off;
      const long long out_ext = p.ext[half == 0 ? kTdv : kTdk];   // debug bounds checks
      constexpr int kChunks = D / 8;                   // 16-byte chunks per row
      constexpr int kRowsPer = 32 / kChunks;           // rows per store instruction
      auto sw = [](int rr) { return kChunks >= 8 ? (rr & 7) : ((rr >> 1) & 3); };
      static_assert(32 * D * 2 <= 4096 && 8 * 4096 <= C::kPBytes, "the dS^T buffer holds them");
      // a warp's dS^T rows are 4 KB of the buffer at warp * 4 KB (32 key rows
      // of one 128-byte column block)
      const uint32_t stage = sDST + warp * 4096;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + col0 + cc * 32, o);
        tmem_ld_wait();
        if (cc == D / 32 - 1) {
          // dV / dK read out: the next item's first dV / dK may overwrite them
          tc_fence_before();
          mbar_arrive(&bars->acc_free);
        }
        if (nsteps == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int chunk = cc * 4 + e;
          st_shared_v4(stage + (lane * kChunks + (chunk ^ sw(lane))) * 16,
                       Pack2<T>::pack(__uint_as_float(o[8 * e + 0]) * sc, __uint_as_float(o[8 * e + 1]) * sc),
                       Pack2<T>::pack(__uint_as_float(o[8 * e + 2]) * sc, __uint_as_float(o[8 * e + 3]) * sc),
                       Pack2<T>::pack(__uint_as_float(o[8 * e + 4]) * sc, __uint_as_float(o[8 * e + 5]) * sc),
                       Pack2<T>::pack(__uint_as_float(o[8 * e + 6]) * sc, __uint_as_float(o[8 * e + 7]) * sc));
        }
      }
      __syncwarp();
      const int c = lane % kChunks;
      const long long base = reinterpret_cast<long long>(out);
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int rr = i * kRowsPer + lane / kChunks;  // the row whose chunk c this lane stores
        const T* dst = reinterpret_cast<const T*>(__shfl_sync(0xffffffffu, base, rr));
        const long long dst_off = __shfl_sync(0xffffffffu, out_off, rr);
        uint4 w;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w) : "r"(stage + (rr * kChunks + (c ^ sw(rr))) * 16)
                     : "memory");
        if (key - lane + rr < Lk && SDPA_CHECK(dst_off + 8 * c + 8 <= out_ext, p.status))
          *reinterpret_cast<uint4*>(const_cast<T*>(dst) + 8 * c) = w;
      }
      __syncwarp();                                    // the staged rows are read before the next item writes dS^T
     }
     g0 += nsteps;
     ++kv;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaSWarp) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
  }
}

template <int D, typename T, bool CAUSAL, bool PACKED, int EXT>
cudaError_t launch_persist_one(const BwdProblem& bp, const BwdMaps& m, cudaStream_t s) {
  auto kern = bwd_persist_kernel<D, T, CAUSAL, PACKED, EXT>;
  using C = PCfg<D, EXT>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    // setmaxnreg redistributes the registers the block is launched with; a
    // split larger than that would wait forever, so refuse to launch instead
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < static_cast<int>(256 * kRegsSoftmax + 256 * kRegsOther)) return cudaErrorInvalidConfiguration;
    attr_set[dev] = 1;
  }
  const Problem& p = bp.f;
  const long long units = static_cast<long long>(p.B) * p.H;
  const long long blocks = static_cast<long long>((p.Lk + BK - 1) / BK) * units;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdProblem g = bp;
  // causal: as many units per group as keep their Q, dO (2 bytes per element)
  // and dQ accumulator (4) within kL2Budget; without masking every CTA has
  // the same work and the units simply go one after another
  constexpr long long kL2Budget = 48ll << 20;
  const long long unit_bytes = static_cast<long long>(p.cu_seqlens ? p.max_q : p.Lq) * D * 8;
  g.group = p.causal ? static_cast<int>(std::max(1ll, std::min(units, kL2Budget / std::max(1ll, unit_bytes)))) : 1;
  // persistent kernels: one CTA per SM claiming key blocks, each launch with
  // its own scheduler slot (the last claimer resets it)
  static int sm_count[64] = {0};
  static unsigned* sched_base[64] = {nullptr};
  static std::atomic<unsigned> launches{0};
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (sm_count[dev] == 0 && (e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if (sched_base[dev] == nullptr) {
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_bwd_sched)) != cudaSuccess) return e;
    sched_base[dev] = static_cast<unsigned*>(ptr);
  }
  // one CTA per SM claiming key blocks; each launch has its own scheduler
  // slot (the last claimer resets it)
  const unsigned grid = static_cast<unsigned>(std::min<long long>(blocks, sm_count[dev]));
  unsigned* sched = sched_base[dev] + 2 * (launches.fetch_add(1) % kBSchedSlots);
  kern<<<grid, kThreads, C::kSmem, s>>>(g, m.q, m.k, m.v, m.dO, sched);
  return cudaGetLastError();
}


}  // namespace

template <int D, typename T>
cudaError_t launch_bwd_persist(const BwdProblem& bp, const BwdMaps& m, cudaStream_t s) {
  if (bp.f.strided)
    return bp.f.causal ? launch_persist_one<D, T, true, false, 4>(bp, m, s) : launch_persist_one<D, T, false, false, 4>(bp, m, s);
  if (bp.f.cu_seqlens != nullptr) return cudaErrorNotSupported;   // packed batches: bwd_tc.cu
  return bp.f.causal ? launch_persist_one<D, T, true, false, 0>(bp, m, s) : launch_persist_one<D, T, false, false, 0>(bp, m, s);
}

template cudaError_t launch_bwd_persist<32, __half>(const BwdProblem&, const BwdMaps&, cudaStream_t);
template cudaError_t launch_bwd_persist<64, __half>(const BwdProblem&, const BwdMaps&, cudaStream_t);
template cudaError_t launch_bwd_persist<32, __nv_bfloat16>(const BwdProblem&, const BwdMaps&, cudaStream_t);
template cudaError_t launch_bwd_persist<64, __nv_bfloat16>(const BwdProblem&, const BwdMaps&, cudaStream_t);

}  // namespace sdpa
