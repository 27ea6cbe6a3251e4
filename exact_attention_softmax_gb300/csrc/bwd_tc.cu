// bwd_tc.cu -- exact attention backward on the sm_103a tensor cores.
//
// Recomputation as in the FlashAttention news article (QbitAI repost, section
// "FlashAttention"): the probabilities are rebuilt from Q, K and the saved
// log-sum-exp rather than stored. Each CTA keeps one 128-key block of K and V
// (and its dK, dV accumulators in TMEM) and streams the query tiles that can
// see it. Per query tile i of BQ rows, with keys on TMEM lanes:
//
//   S^T  = K Q_i^T,  dP^T = V dO_i^T                          (tcgen05, TMEM)
//   P^T  = exp(scale S^T - LSE_i)                              (CUDA cores -> TMEM)
//   dS^T = P^T * (dP^T - D_i)                                  (CUDA cores -> SMEM)
//   dV  += P^T dO_i  (A from TMEM);  dK += dS^T Q_i            (tcgen05, TMEM)
//   dQ_i partial = dS K   (d <= 64: M = query rows)
//             or  (K^T dS^T)^T (d = 128: M = head dims)       (tcgen05, TMEM)
//
// and the dQ partial is added into an fp32 accumulator in global memory (one
// bulk shared->global reduce per tile at d = 128, vector reductions of whole
// row segments at d <= 64). dK = scale * dK_acc and dV are written at the
// end; dQ = scale * dQ_acc is rounded by a separate kernel.
//
// Warps: 0-3 and 4-7 build P^T / dS^T for the first and second half of the
// tile's queries (then write dV and dK); 8-11 drain dQ; 12 loads with TMA;
// 13 issues S^T and dP^T (and dQ at d <= 64); 14 issues dV and dK (and dQ at
// d = 128); 15 loads the additive mask (masked kernels; it idles otherwise).
// The softmax groups release S^T / dP^T as soon as they hold them in
// registers, so the next tile's S^T, dP^T run under their arithmetic. P^T
// goes to TMEM, where the dV MMA reads it, so only dS^T passes through shared
// memory (whose bandwidth the MMAs' operand reads also use); the one dQ
// buffer is drained well within a step. At d = 128 two handoffs inside a step
// are split: S^T and dP^T commit separately, so P is formed while the dP^T
// MMAs run, and P^T reaches the dV MMA before dS is formed.
#include <algorithm>

#include "bwd_common.cuh"

namespace sdpa {
namespace {

// EXT (dense layout only): 0 plain, 1 block-sparse (p.bmask), 2 additive mask
// (p.amask), 3 dropout (p.dropout), 4 plain on strided tensors (p.strided).
template <int D, typename T, bool CAUSAL, bool PACKED, int EXT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const BwdProblem bp, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmM) {
  using C = BCfg<D, EXT>;
  constexpr bool SPARSE = EXT == 1, BIAS = EXT == 2, DROP = EXT == 3, STRIDED = EXT == 4;
  constexpr int BQ = C::BQ;
  constexpr int NH = C::kHalf;     // query columns per softmax group
  // The additive mask and dropout need registers of their own, so their
  // steps go through in chunks of 32 query columns (S^T / dP^T read from
  // TMEM a chunk at a time); the other kernels take the half in one piece.
  constexpr int CH = (BIAS || DROP) && NH > 32 ? 32 : NH;
  constexpr int NCH = NH / CH;
  // P from S^T before dP^T is read, and P^T handed to the dV MMA before dS^T
  // is formed (one chunk of at most 32 columns: d = 128)
  constexpr bool kSplitDP = NCH == 1 && CH <= 32;
  static_assert(!kSplitDP || C::kDsTmem, "the split path stores dS^T in TMEM");
  static_assert(!BIAS || CH * BK * 2 == C::kMaskTile, "a mask slot holds one chunk of each softmax group");
  const Problem& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + C::kOffBar);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Packed batches: a unit is (sequence, head); its queries are rows
  // cu_seqlens[s] .. cu_seqlens[s+1]-1 of the query token axis, its keys rows
  // cu_k[s] .. cu_k[s+1]-1 of the key token axis, and p.Lk bounds every key length.
  const int nkb = (p.Lk + BK - 1) / BK;
  // CTAs go out in groups of bp.group units; inside a group key block 0 of
  // every unit comes first, then key block 1, and so on. Under causal masking
  // low key blocks see the most query rows, so the longest CTAs start first,
  // while a group's Q, dO and dQ accumulator stay small enough for L2.
  const int per_group = bp.group * nkb;
  const int grp = blockIdx.x / per_group, rg = blockIdx.x % per_group;
  const int gunits = min(bp.group, p.B * p.H - grp * bp.group);
  const int unit = grp * bp.group + rg % gunits;
  const int kblk = rg / gunits;
  const int key0 = kblk * BK;
  int Lq = p.Lq, Lk = p.Lk, tok0 = 0, tok0k = 0, head = 0;
  if (PACKED) {
    const int sq = unit / p.H;
    head = unit % p.H;
    tok0 = p.cu_seqlens[sq];
    Lq = p.cu_seqlens[sq + 1] - tok0;
    tok0k = p.cu_k[sq];
    Lk = p.cu_k[sq + 1] - tok0k;
    const bool bad = Lq > p.max_q || Lk > p.Lk || (Lq > 0 && Lk <= 0);
    if (bad && kblk == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
    if (bad) return;  // lengths outside their bounds: reported, nothing written
  }
  if (key0 >= Lk) return;
  // element offset of row 0 of this unit (query side, key side), stride between
  // rows, and offset of its row statistics (dense: [B,H,L,d] and [B,H,L];
  // packed: [total,H,d] and [H,total])
  const long long row0 = PACKED ? (static_cast<long long>(tok0) * p.H + head) * D : 0;
  const long long row0k = PACKED ? (static_cast<long long>(tok0k) * p.H + head) * D : 0;
  const long long rstride = PACKED ? static_cast<long long>(p.H) * D : D;
  const long long stat0 = PACKED ? static_cast<long long>(head) * p.Lq + tok0 : static_cast<long long>(unit) * Lq;
  const int nq = (Lq + BQ - 1) / BQ;
  const int i0 = CAUSAL ? min(nq, key0 / BQ) : 0;
  // Block-sparse (dense layout): only the query steps whose 128-row mask
  // block keeps this key block run; one warp lists them before the roles start.
  constexpr bool sparse = SPARSE;
  uint16_t* slist = reinterpret_cast<uint16_t*>(smem + C::kOffList);

  const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sDST = smem_u32(smem + C::kOffDST);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);   // [stage][2][BQ]

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv, 1);
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
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->kv_done, 1);
    mbar_init(&bars->done, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->mfull[i], 1);
      mbar_init(&bars->mempty[i], 8);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (sparse && warp == 1) {
    const unsigned char* mcol = p.bmask + (unit / p.H) * p.bm_sb + (unit % p.H) * p.bm_sh + kblk;
    int cnt = 0;
    for (int base = i0; base < nq; base += 32) {
      const int qi = base + lane;
      const bool act = qi < nq && mcol[static_cast<long long>(qi * BQ / kMaskBlock) * p.bm_sq] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, act);
      const int at = cnt + __popc(bal & ((1u << lane) - 1u));
      if (act && at < C::kMaxSteps) slist[at] = static_cast<uint16_t>(qi);
      cnt += __popc(bal);
    }
    if (lane == 0) bars->nsteps = min(cnt, C::kMaxSteps);
  }
  if (warp == kMmaSWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile uint32_t* abort_flag = &bars->abort_flag;
  const int nsteps = sparse ? bars->nsteps : nq - i0;
  // query step (in BQ rows) of the CTA's s-th step
  auto qstep = [&](int st) { return sparse ? (st < nsteps ? static_cast<int>(slist[st]) : nq) : i0 + st; };
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
    // boxes: packed (column, head, token); dense (column, row, unit), or
    // (column, row, head, batch) through 4-D maps of strided tensors
    auto load = [&](void* dst, const CUtensorMap* m, uint64_t* bar, int col, int row, int tok) {
      if constexpr (PACKED) tma_load_3d(dst, m, bar, col, head, tok + row);
      else if constexpr (STRIDED) tma_load_4d(dst, m, bar, col, row, unit % p.H, unit / p.H);
      else tma_load_3d(dst, m, bar, col, row, unit);
    };
    if (lane == 0 && !*abort_flag) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_expect_tx(&bars->kv, 2 * C::kKTile);
      for (int cb = 0; cb < C::kNBlk; ++cb) {
        load(smem + C::kOffK + cb * C::kKColBlk, &tmK, &bars->kv, cb * C::kBlk, key0, tok0k);
        load(smem + C::kOffV + cb * C::kKColBlk, &tmV, &bars->kv, cb * C::kBlk, key0, tok0k);
      }
    }
    const float* lse = p.lse + stat0;
    const float* delta = bp.delta + stat0;
    // The row statistics of step s + 1 are fetched into registers while step s
    // is in flight, so their latency hides behind the wait for a free stage.
    constexpr int kPer = BQ / 32;
    float nl[kPer], nd[kPer];
    auto fetch = [&](int step) {
      const int q0 = qstep(step) * BQ;
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
      const int stage = s % C::kStages, round = s / C::kStages;
      bool ok = !*abort_flag;
      if (ok && lane == 0 && round > 0) ok = mbar_wait(&bars->empty[stage], (round - 1) & 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const int q0 = qstep(s) * BQ;
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
    if (lane == 0 && *abort_flag) {
      mbar_wait_drain(&bars->kv, 0);
      for (int f = max(0, s - C::kStages); f < s; ++f) mbar_wait_drain(&bars->full[f % C::kStages], (f / C::kStages) & 1);
    }
   } else if (warp == kMmaSWarp || warp == kMmaGWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __half>::value ? 0u : 1u;
      auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort_flag, p.status); };
      bool ok = wait(&bars->kv, 0);
      // dQ partial of tile t: contraction over the 128 keys, both operands MN-major
      constexpr uint32_t idQ = C::kDqT ? idesc_f16(fmt, 1, 1, D, BQ)    // dQ^T: M = D, N = queries
                                       : idesc_f16(fmt, 1, 1, BQ, D);   // dQ: M = queries, N = D
      const uint64_t dKm = smem_desc(sK, C::kKColBlk, C::kSbo, C::kSw);
      const uint64_t dDSm = smem_desc(sDST, C::kPColBlk, 1024, kSwizzle128B);
      auto issue_dq = [&](int t) {
        if (!wait(&bars->pds_full, t & 1)) return false;
        const int buf = 0;
        if (t >= 1 && !wait(&bars->dq_free[0], (t - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t tdq = tmem + C::kTdQ + buf * C::kDqCols;
        // contraction over the 128 keys, both operands MN-major
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint32_t kb_off = (ks * 16 * C::kRowBytes) >> 4;   // 16 key rows of the K tile
          const uint32_t ds_off = (ks * 16 * 128) >> 4;            // 16 key rows of dS^T
          if (C::kDqT) mma_ss(tdq, dKm + kb_off, dDSm + ds_off, idQ, ks > 0);
          else mma_ss(tdq, dDSm + ds_off, dKm + kb_off, idQ, ks > 0);
        }
        mma_commit(&bars->dq_full[buf]);
        mma_commit(&bars->pds_free);
        return true;
      };
      if (warp == kMmaSWarp) {
        // S^T = K Q^T and dP^T = V dO^T (K-major operands, contraction over D),
        // and the dQ partial of the previous tile
        constexpr uint32_t idS = idesc_f16(fmt, 0, 0, BK, BQ);

        const uint64_t dK0 = smem_desc(sK, 16, C::kSbo, C::kSw);
        const uint64_t dV0 = smem_desc(sV, 16, C::kSbo, C::kSw);
        const uint64_t dQ0 = smem_desc(sQ, 16, C::kSbo, C::kSw);
        const uint64_t dO0 = smem_desc(sDO, 16, C::kSbo, C::kSw);
        for (int s = 0; s < nsteps && ok; ++s) {
          const int stage = s % C::kStages;
          if (!(ok = wait(&bars->full[stage], (s / C::kStages) & 1))) break;
          if (s > 0 && !(ok = wait(&bars->s_free, (s - 1) & 1))) break;
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
          // dQ of the previous tile: needs its dS^T and a free dQ buffer
          if (C::kDqOnS && s > 0 && !(ok = issue_dq(s - 1))) break;
        }
        if (C::kDqOnS && ok && nsteps > 0) ok = issue_dq(nsteps - 1);
      } else {
        // dV += P^T dO, dK += dS^T Q (A K-major over queries, B MN-major)
        constexpr uint32_t idKV = idesc_f16(fmt, 0, 1, BK, D);
        const uint64_t dDST = smem_desc(sDST, 16, 1024, kSwizzle128B);
        const uint64_t dQm = smem_desc(sQ, C::kQColBlk, C::kSbo, C::kSw);
        const uint64_t dOm = smem_desc(sDO, C::kQColBlk, C::kSbo, C::kSw);
        for (int s = 0; s < nsteps && ok; ++s) {
          const int stage = s % C::kStages;
          const uint32_t qoff = (stage * C::kQTile) >> 4;
          if constexpr (kSplitDP) {
            // dV as soon as P^T is in TMEM, then dK once dS^T is
            if (!(ok = wait(&bars->p_full, s & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks)
              mma_ts(tmem + C::kTdV, tmem + C::kTP + ks * 8, dOm + qoff + ((ks * 16 * C::kRowBytes) >> 4), idKV,
                     (s > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&bars->p_free);
            if (!(ok = wait(&bars->pds_full, s & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks)
              mma_ts(tmem + C::kTdK, tmem + C::kTDS + ks * 8, dQm + qoff + ((ks * 16 * C::kRowBytes) >> 4), idKV,
                     (s > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&bars->pds_free);
            mma_commit(&bars->empty[stage]);
            if (!C::kDqOnS && !(ok = issue_dq(s))) break;
            continue;
          }
          if (!(ok = wait(&bars->pds_full, s & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < BQ / 16; ++ks) {
            const uint32_t aoff = ((ks / 4) * C::kPColBlk + (ks % 4) * 32) >> 4;
            const uint32_t boff = qoff + ((ks * 16 * C::kRowBytes) >> 4);
            const uint32_t acc = (s > 0 || ks > 0) ? 1u : 0u;
            mma_ts(tmem + C::kTdV, tmem + C::kTP + ks * 8, dOm + boff, idKV, acc);
            if constexpr (C::kDsTmem) mma_ts(tmem + C::kTdK, tmem + C::kTDS + ks * 8, dQm + boff, idKV, acc);
            else mma_ss(tmem + C::kTdK, dDST + aoff, dQm + boff, idKV, acc);
          }
          mma_commit(&bars->pds_free);
          mma_commit(&bars->empty[stage]);
          if (!C::kDqOnS && !(ok = issue_dq(s))) break;
        }
        mma_commit(&bars->kv_done);
      }
      mma_commit(&bars->done);
      mbar_wait_drain(&bars->done, 0);
    }
   } else if (BIAS && warp == kMaskWarp) {
    // ------------------------------------------------ additive mask loads
    // Chunk n (query step n / NCH, columns (n % NCH) * CH of each group) goes
    // to slot n % 2 as one 32 x 128 box per softmax group, so the mask of the
    // next chunk is in flight while a chunk computes.
    if (lane == 0 && !*abort_flag) {
      tma_prefetch_desc(&tmM);
      const int zc = p.am_sh ? unit % p.H : 0, wc = p.am_sb ? unit / p.H : 0;
      const int total = nsteps * NCH;
      int n = 0;
      for (; n < total; ++n) {
        const int slot = n & 1;
        if (n >= 2 && !mbar_wait(&bars->mempty[slot], ((n - 2) >> 1) & 1, abort_flag, p.status)) break;
        const int q0 = qstep(n / NCH) * BQ + (n % NCH) * CH;
        mbar_expect_tx(&bars->mfull[slot], C::kMaskSlot);
        for (int h = 0; h < 2; ++h)
          tma_load_4d(smem + C::kOffList + slot * C::kMaskSlot + h * C::kMaskTile, &tmM, &bars->mfull[slot], key0,
                      q0 + h * NH, zc, wc);
      }
      if (*abort_flag)
        for (int f = max(0, n - 2); f < n; ++f) mbar_wait_drain(&bars->mfull[f & 1], (f >> 1) & 1);
    }
   } else if (warp < kDqWarp0 + 4) {
    // ------------------------------------------------ dQ drain
    // d = 128 (lane = head dim, columns = queries): staged as [query][D] in
    // shared memory and added with one bulk shared->global reduce per tile.
    // d = 64 (lane = query row): 16-byte vector reductions straight from the
    // registers, which spares shared memory (the backward is bound by its
    // bandwidth); with lane = head dim those would be scalar and slower.
    const int r = threadIdx.x & 127;                          // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const long long dq_base = PACKED ? row0 : static_cast<long long>(unit) * Lq * D;
    float* dq_unit = bp.dq_acc + dq_base;
    const long long dq_ext = bp.acc_rows * D;   // elements of the accumulator (debug bounds checks)
    const uint32_t sDQ = smem_u32(smem + C::kOffDQ);
    for (int s = 0; s < nsteps; ++s) {
      const int buf = 0;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dq_full[0], s & 1, abort_flag, p.status))) break;
      tc_fence_after();
      const int q0 = qstep(s) * BQ;
      const uint32_t tdq = tmem + lane_off + C::kTdQ + buf * C::kDqCols;
      if (C::kDqT) {
        if (r == 0) bulk_wait_read0();          // the previous reduce has read the staging tile
        named_bar_sync(1, 128);
#pragma unroll 1
        for (int cc = 0; cc < BQ / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tdq + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) st_shared_f32(sDQ + ((cc * 32 + e) * D + r) * 4, __uint_as_float(o[e]));
        }
        tc_fence_before();
        mbar_arrive(&bars->dq_free[buf]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (r == 0) {
          const int rows = min(BQ, Lq - q0);
          if (!PACKED) {
            if (SDPA_CHECK(dq_base + static_cast<long long>(q0 + rows) * D <= dq_ext, p.status))
              bulk_reduce_add_f32(dq_unit + static_cast<long long>(q0) * D, sDQ, static_cast<uint32_t>(rows * D * 4));
          } else {
            // packed rows are H * D apart: one reduce per row
            for (int q = 0; q < rows; ++q)
              if (SDPA_CHECK(dq_base + static_cast<long long>(q0 + q) * rstride + D <= dq_ext, p.status))
                bulk_reduce_add_f32(dq_unit + static_cast<long long>(q0 + q) * rstride, sDQ + q * D * 4, D * 4);
          }
          bulk_commit();
        }
      } else {
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
    }
    if (C::kDqT && r == 0) bulk_wait0();
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------ P^T and dS^T, then dV / dK
    const int half = warp / 4;                                // query columns [half * kHalf, +kHalf)
    const int r = threadIdx.x & 127;                          // key row == TMEM lane
    const int key = key0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale * kLog2e;
    bool ok = true;
    // this thread's key column of the additive mask slots ([32 queries][128 keys] per group)
    const T* mkey = reinterpret_cast<const T*>(smem + C::kOffList + half * C::kMaskTile) + r;
    for (int s = 0; s < nsteps; ++s) {
      const int stage = s % C::kStages;
      // With one chunk of at most 32 columns (d = 128) P is computed from S^T
      // while the dP^T MMAs run, and dP^T is loaded after it; otherwise (the
      // 64 columns of d <= 64 would then spill) both are loaded together.
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, s & 1, abort_flag, p.status) &&
                                       mbar_wait(&bars->full[stage], (s / C::kStages) & 1, abort_flag, p.status) &&
                                       (kSplitDP || mbar_wait(&bars->dp_full, s & 1, abort_flag, p.status)));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[NCH][CH], dv[NCH][CH];
#pragma unroll
      for (int cc = 0; cc < CH / 32; ++cc) {
        tmem_ld32(tmem + lane_off + C::kTS + half * NH + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[0][cc * 32]));
        if (!kSplitDP)
          tmem_ld32(tmem + lane_off + C::kTdP + half * NH + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[0][cc * 32]));
      }
      tmem_ld_wait();
      if (NCH == 1 && !kSplitDP) {
        tc_fence_before();
        mbar_arrive(&bars->s_free);             // the next S^T / dP^T may be written
      }
      const int qh = qstep(s) * BQ + half * NH;  // this group's first query column
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int q0 = qh + ch * CH;
        const bool need_mask = (CAUSAL && q0 < key0 + BK - 1) || (key0 + BK > Lk);
        // dropout: the 16 keys of a half-warp share one Philox block per
        // query; lane o of the half computes the blocks of columns o and
        // o + 16, and a byte transpose hands every lane its own bytes
        uint32_t dw[DROP ? CH / 16 : 1][4];
        if (DROP) {
          const int hl = threadIdx.x & 15;
#pragma unroll
          for (int t = 0; t < CH / 16; ++t) {
            const uint4 rv = philox4x32_10(make_uint4(static_cast<uint32_t>(key >> 4), static_cast<uint32_t>(q0 + hl + 16 * t),
                                                      static_cast<uint32_t>(unit), 0u),
                                           p.seed_lo, p.seed_hi);
            dw[t][0] = rv.x; dw[t][1] = rv.y; dw[t][2] = rv.z; dw[t][3] = rv.w;
            transpose16_bytes(dw[t], hl);
          }
        }
        // additive mask of this chunk, staged in slot n % 2 by the mask warp
        const int n = s * NCH + ch;
        const T* mt = mkey + (n & 1) * (C::kMaskSlot / 2);
        if (BIAS) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->mfull[n & 1], (n >> 1) & 1, abort_flag, p.status));
          if (!ok) break;
        }
        uint32_t pk[CH / 2], dk[CH / 2];
        // row statistics of these query columns (written by the producer
        // before it arrived on full[stage])
        const float* slf = stat + stage * 2 * BQ + half * NH + ch * CH;
        // dropout factor of (query q0 + col, key)
        auto zf_of = [&](int col) {
          if (!DROP) return 1.f;
          const uint32_t byte = __byte_perm(dw[col >> 4][(col & 15) >> 2], 0u, 0x4440u | (col & 3));
          return byte >= p.drop_t ? p.drop_scale : 0.f;
        };
        // P of this chunk, kept (as bits, in place of S) for dS and packed
        // for P^T; the per-element causal / length test only where the tile
        // needs it
        auto body_p = [&](auto masked) {
          constexpr bool M = decltype(masked)::value;
#pragma unroll
          for (int g = 0; g < CH / 4; ++g) {
            // loaded in program order: hoisting them costs registers and spills
            float l4[4];
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(l4[0]), "=f"(l4[1]), "=f"(l4[2]), "=f"(l4[3]) : "r"(smem_u32(slf + 4 * g)));
            float pr[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int col = 4 * g + h;
              // P = 2^(S * scale * log2(e) - LSE2); with a mask S * scale + M
              // is formed first, in natural-log units. (The plain d = 64
              // kernels keep the addend as a subtraction: with the negated
              // operand ptxas spills there and they measured slower.)
              const float s_ = __uint_as_float(sv[ch][col]);
              float pv;
              if (BIAS) pv = ex2_approx(fmaf(fmaf(s_, p.scale, to_f32(mt[col * BK])), kLog2e, -l4[h]));
              else if (D == 128 || DROP) pv = ex2_approx(fmaf(s_, c, -l4[h]));
              else pv = ex2_approx(fmaf(s_, c, 0.f - l4[h]));
              if (M && ((CAUSAL && q0 + col < key) || key >= Lk)) pv = 0.f;
              sv[ch][col] = __float_as_uint(pv);
              pr[h] = pv * zf_of(col);
            }
            pk[2 * g] = Pack2<T>::pack(pr[0], pr[1]);
            pk[2 * g + 1] = Pack2<T>::pack(pr[2], pr[3]);
          }
        };
        // P and dS together (when dP^T is already in registers)
        auto body = [&](auto masked) {
          constexpr bool M = decltype(masked)::value;
#pragma unroll
          for (int g = 0; g < CH / 4; ++g) {
            // loaded in program order: hoisting them costs registers and spills
            float l4[4], d4[4];
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(l4[0]), "=f"(l4[1]), "=f"(l4[2]), "=f"(l4[3]) : "r"(smem_u32(slf + 4 * g)));
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(d4[0]), "=f"(d4[1]), "=f"(d4[2]), "=f"(d4[3]) : "r"(smem_u32(slf + BQ + 4 * g)));
            float pr[4], ds[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int col = 4 * g + h;
              const float s_ = __uint_as_float(sv[ch][col]);
              float pv;
              if (BIAS) pv = ex2_approx(fmaf(fmaf(s_, p.scale, to_f32(mt[col * BK])), kLog2e, -l4[h]));
              else if (D == 128 || DROP) pv = ex2_approx(fmaf(s_, c, -l4[h]));
              else pv = ex2_approx(fmaf(s_, c, 0.f - l4[h]));
              if (M && ((CAUSAL && q0 + col < key) || key >= Lk)) pv = 0.f;
              const float zf = zf_of(col);
              pr[h] = pv * zf;
              ds[h] = pv * (__uint_as_float(dv[ch][col]) * zf - d4[h]);
            }
            pk[2 * g] = Pack2<T>::pack(pr[0], pr[1]);
            pk[2 * g + 1] = Pack2<T>::pack(pr[2], pr[3]);
            dk[2 * g] = Pack2<T>::pack(ds[0], ds[1]);
            dk[2 * g + 1] = Pack2<T>::pack(ds[2], ds[3]);
          }
        };
        // dS = P * (dP - D) of this chunk (dropout: P * (dP * z - D)), packed
        auto body_ds = [&]() {
#pragma unroll
          for (int g = 0; g < CH / 4; ++g) {
            float d4[4];
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(d4[0]), "=f"(d4[1]), "=f"(d4[2]), "=f"(d4[3]) : "r"(smem_u32(slf + BQ + 4 * g)));
            float ds[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int col = 4 * g + h;
              ds[h] = __uint_as_float(sv[ch][col]) * (__uint_as_float(dv[ch][col]) * zf_of(col) - d4[h]);
            }
            dk[2 * g] = Pack2<T>::pack(ds[0], ds[1]);
            dk[2 * g + 1] = Pack2<T>::pack(ds[2], ds[3]);
          }
        };
        if constexpr (!kSplitDP) {
          if (need_mask) body(std::true_type{});
          else body(std::false_type{});
        } else {
          if (need_mask) body_p(std::true_type{});
          else body_p(std::false_type{});
          // P^T into TMEM once the previous step's dV MMAs have read it, so
          // this step's dV runs while dS is formed
          if (s > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_free, (s - 1) & 1, abort_flag, p.status));
          if (!ok) break;
          {
            const uint32_t tp = tmem + lane_off + C::kTP + (half * NH) / 2;
#pragma unroll
            for (int x = 0; x < CH / 32; ++x) tmem_st16(tp + x * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * x]));
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full);
          // dP^T, whose MMAs ran while P was computed
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full, s & 1, abort_flag, p.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < CH / 32; ++cc)
            tmem_ld32(tmem + lane_off + C::kTdP + half * NH + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[0][cc * 32]));
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars->s_free);             // the next S^T / dP^T may be written
          body_ds();
        }
        if (BIAS) {
          __syncwarp();
          if ((threadIdx.x & 31) == 0) mbar_arrive(&bars->mempty[n & 1]);   // slot read
        }
        if (ch + 1 < NCH) {
          // the next chunk's S^T / dP^T; after the last one TMEM is free
#pragma unroll
          for (int cc = 0; cc < CH / 32; ++cc) {
            const int col = half * NH + (ch + 1) * CH + cc * 32;
            tmem_ld32(tmem + lane_off + C::kTS + col, *reinterpret_cast<uint32_t(*)[32]>(&sv[ch + 1][cc * 32]));
            tmem_ld32(tmem + lane_off + C::kTdP + col, *reinterpret_cast<uint32_t(*)[32]>(&dv[ch + 1][cc * 32]));
          }
          tmem_ld_wait();
          if (ch + 1 == NCH - 1) {
            tc_fence_before();
            mbar_arrive(&bars->s_free);
          }
        }
        // P^T / dS^T buffers are free once the previous tile's dV, dK, dQ MMAs finished
        if (ch == 0 && s > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->pds_free, (s - 1) & 1, abort_flag, p.status));
        if (!ok) break;
        // P^T (and at d = 128 dS^T) into TMEM, this thread's key row, two
        // queries per column; dS^T into shared memory: [key row][query] in
        // 128-byte swizzled rows, 64 queries per column block
        {
          const uint32_t tp = tmem + lane_off + C::kTP + (half * NH + ch * CH) / 2;
          if constexpr (C::kDsTmem) {
            const uint32_t td = tmem + lane_off + C::kTDS + (half * NH + ch * CH) / 2;
#pragma unroll
            for (int x = 0; x < CH / 32; ++x) {
              if (!kSplitDP) tmem_st16(tp + x * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * x]));
              tmem_st16(td + x * 16, *reinterpret_cast<const uint32_t(*)[16]>(&dk[16 * x]));
            }
          } else if constexpr (CH == 64) {
            tmem_st32(tp, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
          } else {
#pragma unroll
            for (int x = 0; x < CH / 32; ++x) tmem_st16(tp + x * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * x]));
          }
        }
#pragma unroll
        for (int c8 = 0; c8 < CH / 8; ++c8) {
          const int chunk = half * (NH / 8) + ch * (CH / 8) + c8;   // 8-query chunk index within the tile
          const uint32_t off = (chunk / 8) * C::kPColBlk + r * 128 + (((chunk % 8) ^ (r & 7)) << 4);
          st_shared_v4(sDST + off, dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2], dk[4 * c8 + 3]);
        }
      }
      if (!ok) break;
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bars->pds_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_done, 0, abort_flag, p.status));
    if (ok) {
      // group 0 writes dV, group 1 writes dK = scale * dK_acc. Every MMA that
      // read the Q/dO stages has finished (kv_done), so each warp stages its
      // 32 rows there (16-byte chunk c of row r at slot c ^ f(r), f(r) = r % 8,
      // or (r / 2) % 4 for the 4-chunk rows of d = 32: the 8 lanes of a
      // quarter-warp hit 8 different bank groups) and stores them back whole
      // rows per instruction instead of 32 rows of 16 bytes.
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
      static_assert(8 * 32 * D * 2 <= 2 * C::kStages * C::kQTile, "the Q/dO stages hold the staged rows");
      const uint32_t stage = smem_u32(smem + C::kOffQ + warp * 32 * D * 2);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + col0 + cc * 32, o);
        tmem_ld_wait();
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
cudaError_t launch_one(const BwdProblem& bp, const BwdMaps& m, cudaStream_t s) {
  auto kern = bwd_tc_kernel<D, T, CAUSAL, PACKED, EXT>;
  using C = BCfg<D, EXT>;
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
  kern<<<static_cast<unsigned>(blocks), kThreads, C::kSmem, s>>>(g, m.q, m.k, m.v, m.dO, m.mask);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_d(const BwdProblem& bp, const BwdMaps& m, cudaStream_t s) {
  if (bp.f.bmask != nullptr)
    return bp.f.causal ? launch_one<D, T, true, false, 1>(bp, m, s) : launch_one<D, T, false, false, 1>(bp, m, s);
  if (bp.f.amask != nullptr)
    return bp.f.causal ? launch_one<D, T, true, false, 2>(bp, m, s) : launch_one<D, T, false, false, 2>(bp, m, s);
  if (bp.f.dropout)
    return bp.f.causal ? launch_one<D, T, true, false, 3>(bp, m, s) : launch_one<D, T, false, false, 3>(bp, m, s);
  // d <= 64 dense or strided, without mask or dropout: persistent CTAs
  // (bwd_persist.cu). Packed batches stay here: their units are short (a few
  // query steps per key block) and one CTA per key block measured faster.
  if constexpr (D <= 64)
    if (bp.f.cu_seqlens == nullptr) return launch_bwd_persist<D, T>(bp, m, s);
  if (bp.f.strided)
    return bp.f.causal ? launch_one<D, T, true, false, 4>(bp, m, s) : launch_one<D, T, false, false, 4>(bp, m, s);
  if (bp.f.cu_seqlens != nullptr)
    return bp.f.causal ? launch_one<D, T, true, true, 0>(bp, m, s) : launch_one<D, T, false, true, 0>(bp, m, s);
  return bp.f.causal ? launch_one<D, T, true, false, 0>(bp, m, s) : launch_one<D, T, false, false, 0>(bp, m, s);
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdProblem& bp, int dtype, const BwdMaps& m, cudaStream_t s) {
  if (dtype == kF16) {
    if (bp.f.d == 32) return launch_d<32, __half>(bp, m, s);
    if (bp.f.d == 64) return launch_d<64, __half>(bp, m, s);
    if (bp.f.d == 128) return launch_d<128, __half>(bp, m, s);
  } else if (dtype == kBF16) {
    if (bp.f.d == 32) return launch_d<32, __nv_bfloat16>(bp, m, s);
    if (bp.f.d == 64) return launch_d<64, __nv_bfloat16>(bp, m, s);
    if (bp.f.d == 128) return launch_d<128, __nv_bfloat16>(bp, m, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace sdpa
