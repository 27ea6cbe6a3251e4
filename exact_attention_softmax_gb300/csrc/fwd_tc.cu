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
//   warp 8      TMA producer: Q tiles, then K_j, V_j into a ring of slots,
//               streaming from one work item into the next
//   warps 9-10  MMA issuers (one thread each; one warp per Q tile for d <= 64,
//               warp 9 alone for d = 128): S_t = Q_t K_j^T and O_t += P_t V_j
//               as tcgen05.mma with fp32 accumulators in TMEM
//   warps 0-3   softmax for tile 0: one thread per query row reads its S row
//   warps 4-7   softmax for tile 1    from TMEM, masks, updates the running max
//               m and sum l, writes P (fp16/bf16) back to TMEM, rescales its
//               O row in TMEM when m grew past a threshold, and finally
//               writes O = O/l and LSE = (m + log2 l) ln 2.
//
// A softmax group releases S_t as soon as it holds the row in registers, so
// Q_t K_{j+1}^T runs under its exponentials, and P.V reads P straight from
// TMEM. For d <= 64 each CTA is persistent and takes work items from a
// dynamic queue: Q is double-buffered, the next item's first S_t is issued
// while the current item's last block is still in its softmax, and the
// current item's epilogue is deferred into the next item's first block, so
// consecutive items overlap instead of draining the pipeline. The d <= 64
// block-sparse kernel splits each CTA into two such pipelines, one per tile
// slot (warp 11 is the second producer), each claiming single 128-row tiles
// and streaming only the key blocks its tile's mask row keeps.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0, O_1 (d each) and P_0, P_1
// (64 columns each) after them; at d = 128 P_t overlays the upper half of S_t.
#include <atomic>
#include <type_traits>

#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 128;          // keys per K/V block
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;      // first MMA warp (also allocates TMEM)
constexpr uint32_t kTmemCols = 512;
// Register split (launch: 384 threads x 168): softmax groups 200, the
// producer / MMA group 104; 256 * 200 + 128 * 104 = 64512 = 384 * 168,
// and per SM sub-partition 200 + 200 + 104 <= 512 registers per lane.
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsControl = 104;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running maximum used in the exponent is only raised when a row's new
// maximum exceeds it by more than this (log2 units), so P <= 2^8 and O is
// rescaled rarely; the result is the same because O and l share the maximum.
constexpr float kRescaleThreshold = 8.0f;

// Dynamic work distribution: each launch takes one slot of {next item, CTAs
// finished}; CTAs claim items with atomicAdd and the last CTA to finish puts
// the slot back to zero. Launches in flight at the same time use different
// slots (a host-side counter walks the slots in turn).
constexpr int kSchedSlots = 1024;
__device__ unsigned g_fwd_sched[2 * kSchedSlots];
constexpr int kItemQueue = 4;
constexpr int kBarBytes = 704;   // shared memory for the barrier block

template <int D, int EXT = 0>
struct Cfg {
  static constexpr int kBlk = D >= 64 ? 64 : D;             // elements per swizzled row
  static constexpr int kNBlk = D / kBlk;                      // column blocks per tile
  static constexpr uint32_t kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kRowBytes = kBlk * 2;                  // 128 or 64
  static constexpr int kSbo = 8 * kRowBytes;                  // 8-row group stride
  static constexpr int kColBlkBytes = 128 * kRowBytes;        // one column block of a 128-row tile
  static constexpr int kTileBytes = 128 * D * 2;              // a Q, K or V tile
  // Q tiles are double-buffered where each CTA runs many work items (d <= 64),
  // so the next item's Q and K/V stream in while the current item finishes.
  static constexpr int kQBufs = D == 128 ? 1 : 2;
  // The additive-mask kernel gives up K/V ring slots at d >= 64 for its mask
  // slots: one 32-row x 128-key slot per softmax warp (two 64-key boxes).
  static constexpr bool kMask = EXT == 2;
  // Where each CTA runs many work items (Q double-buffered, d <= 64) the
  // epilogue stages every softmax warp's 32 output rows in shared memory, so
  // the global stores go out row-contiguous. The dense and dropout kernels
  // stage them in a region of their own, for which d = 64 gives two K/V
  // slots. The block-sparse kernel stages them in the item's own Q buffer
  // instead, which no MMA reads once the item's last P.V has finished (a
  // softmax group's 128 rows of O fill exactly one Q tile): no K/V slot is
  // given up, but the buffer goes back to the producer after the (deferred)
  // epilogue rather than after the item's last S_t, which delays the Q load
  // two items on; that measured slower on the dense causal kernel's short
  // items and on the mask kernel. The mask kernel has no room for a stage
  // region and stores directly, as does d = 128, whose items are long.
  static constexpr bool kStageQ = kQBufs == 2 && EXT == 1;
  static constexpr bool kStageO = kQBufs == 2 && !kStageQ && !kMask;
  static constexpr int kSlots = D == 128 ? (kMask ? 3 : 5) : (D == 64 ? (kMask ? 6 : (kStageO ? 8 : 10)) : 16);
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = 2 * kQBufs * kTileBytes;
  static constexpr int kMaskWarpBytes = 32 * BN * 2;
  static constexpr int kOffMask = kOffSlots + kSlots * kTileBytes;
  static constexpr int kStageWarpBytes = 32 * D * 2;          // 32 rows of O
  static_assert(4 * kStageWarpBytes == kTileBytes, "a softmax group stages one Q tile");
  static constexpr int kOffStage = kOffMask + (kMask ? 8 * kMaskWarpBytes : 0);
  static constexpr int kOffBar = kOffStage + (kStageO ? 8 * kStageWarpBytes : 0);
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;    // barriers + alignment slack
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
  // Block-sparse with an MMA warp per tile (d <= 64): the CTA runs two
  // independent pipelines, one per tile slot, each with its own producer, MMA
  // warp, softmax group, item queue and K/V ring. A slot claims single
  // 128-row tiles and streams only the key blocks that tile's mask row keeps,
  // so tiles keeping many and few blocks balance across slots and CTAs, and
  // neither softmax group idles on a block only the other tile keeps. Each
  // ring is read in order by one MMA warp alone, so that warp never waits on
  // a slot whose previous fill has not landed (which a parity wait could not
  // tell from the fill before that).
  static constexpr bool kTileStreams = EXT == 1 && !kPAlias;
  static constexpr int kRings = kTileStreams ? 2 : 1;
  static constexpr int kRing = kSlots / kRings;                // slots per ring
  // Three warpgroups: two softmax groups and one for the producer and MMA
  // warps (its last warp idles, or with per-tile streams is the second
  // producer), so that registers can move between them.
  static constexpr int kThreads = 384;
  static_assert(kPAlias || kColP + 2 * (BN / 2) <= 512, "TMEM budget");
  static_assert(kRing * kRings == kSlots && kRing >= 3, "ring split");
  static_assert(kSlots <= 16 && kQBufs <= 2, "the barrier arrays hold 16 ring slots and 2 Q buffers per tile");
};

struct __align__(8) Bars {
  uint64_t q_full[4];     // Q_t loaded into buffer b ([t * kQBufs + b])
  uint64_t q_empty[4];    // buffer b may be reloaded: its item's last S_t = Q_t K^T finished, or
                          // (staging in Q) each softmax warp has read its staged rows out
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t s_full[2];     // S_t written by the tensor cores
  uint64_t s_free[2];     // S_t read into registers by its softmax group
  uint64_t p_full[2];     // P_t in TMEM (and O_t rescaled)
  uint64_t pv_done[2];    // O_t += P_t V_j finished
  uint64_t o_free[2];     // O_t read out by the epilogue: the next item may overwrite it
  uint64_t mfull[8];      // additive mask: softmax warp w's slot loaded
  uint64_t item_full[8];  // work-item queues from the producer(s) to the other roles
  uint64_t item_empty[8];  // ([slot * kItemQueue + i]; with a single pipeline only slot 0)
  int item[8];
  int item_n[8];          // per-slot pipelines: blocks the item's tile keeps, counted once by its producer
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Bars) <= kBarBytes, "the barrier block's shared memory");

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

// One work item: 256 query rows (two 128-row tiles) of one (batch|sequence,
// head), or with per-slot pipelines one 128-row tile, described as an item
// whose other tile is empty.
struct Item {
  int unit, h, tok0, tok0k, len_q, len_k, r0, n0, n1, nmax;
  // block-sparse: the two tiles' mask rows and their key-block limits (causal
  // and length); n0, n1, nmax then count the loaded key blocks
  const unsigned char* m0;
  const unsigned char* m1;
  int lim0, lim1;
};

// Block-sparse: a key block is loaded for an item when either tile keeps it
// (within that tile's limit); each tile then processes every loaded block
// below its limit, masking the blocks its own row of the mask drops.
__device__ __forceinline__ bool loaded_block(const Item& it, int j) {
  return (j < it.lim0 && it.m0[j]) || (j < it.lim1 && it.m1[j]);
}
// First key block at or after j that mask row m keeps below lim.
__device__ __forceinline__ int next_kept(const unsigned char* m, int lim, int j) {
  while (j < lim && !m[j]) ++j;
  return j;
}
// Fills of ring r for an item: both tiles' shared stream, or with per-tile
// streams tile r's own kept blocks.
__device__ __forceinline__ int item_fills(const Item& x, bool tiles, int r) {
  return 2 * (!tiles ? x.nmax : r == 0 ? x.n0 : x.n1);
}

// First loaded key block at or after j.
__device__ __forceinline__ int next_loaded(const Item& it, int j) {
  const int lim = max(it.lim0, it.lim1);
  while (j < lim && !loaded_block(it, j)) ++j;
  return j;
}

// Items are numbered unit-major, so the items of one (batch|sequence, head) run
// side by side and share its K/V through L2; under causal masking the longest
// rows of each unit come first.
// nper: items per unit. With TILES item idx is a single 128-row tile run by
// slot `slot`: it is described as tile `slot` of an item whose r0 is that much
// lower, and the other tile keeps nothing; `kept` is the number of key blocks
// its mask row keeps when already known (else -1: counted here).
template <bool CAUSAL, bool PACKED, bool SPARSE, bool TILES = false>
__device__ __forceinline__ Item decode_item(const Problem& p, int idx, int nper, int slot = 0, int kept = -1) {
  Item it;
  // Causal items get shorter with their query position, so they are handed
  // out longest first across all units (ord-major), which keeps the last
  // CTAs to finish from starting long items late. Packed batches go the same
  // way: only long sequences have items at high query positions, and those
  // items are the longest. Dense items without masking all cost the same and
  // the units are taken one after another.
  const int units = p.B * p.H;
  constexpr bool kOrdMajor = CAUSAL || PACKED;
  it.unit = kOrdMajor ? idx % units : idx / nper;
  const int ord = kOrdMajor ? idx / units : idx % nper;
  const int pos = kOrdMajor ? (nper - 1 - ord) : ord;    // pair, or tile, within the unit
  it.h = 0;
  it.tok0 = it.tok0k = 0;
  if (PACKED) {
    const int s = it.unit / p.H;
    it.h = it.unit % p.H;
    it.tok0 = p.cu_seqlens[s];
    it.len_q = p.cu_seqlens[s + 1] - it.tok0;
    it.tok0k = p.cu_k[s];
    it.len_k = p.cu_k[s + 1] - it.tok0k;
    // lengths beyond their bounds, or queries with no keys, are reported
    // (the item is then skipped: its rows stay unwritten)
    const bool bad = it.len_q > p.max_q || it.len_k > p.Lk || (it.len_q > 0 && it.len_k <= 0);
    if (bad && ord == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusSeqlen);
    if (bad) it.len_q = 0;
  } else {
    it.len_q = p.Lq;
    it.len_k = p.Lk;
    // an additive mask shared across the batch: the units of one head run
    // side by side, so the rows of its mask they all read come from L2
    if (p.amask != nullptr && p.am_sb == 0 && p.am_sh != 0 && p.B > 1) it.unit = (it.unit % p.B) * p.H + it.unit / p.B;
  }
  if (TILES) {
    const int rt = pos * BM;
    it.r0 = rt - slot * BM;
    const int n = tile_blocks<CAUSAL>(rt, it.len_q, it.len_k);
    const unsigned char* mrow = p.bmask + (it.unit / p.H) * p.bm_sb + (it.unit % p.H) * p.bm_sh +
                                static_cast<long long>(rt / kMaskBlock) * p.bm_sq;
    int c = kept;              // blocks the tile's mask row keeps
    if (c < 0) {
      c = 0;
      for (int j = 0; j < n; ++j) c += mrow[j] != 0;
    }
    it.m0 = it.m1 = mrow;
    it.lim0 = it.lim1 = c > 0 ? n : 0;
    it.n0 = slot == 0 ? c : 0;
    it.n1 = slot == 1 ? c : 0;
    it.nmax = c;
    return it;
  }
  it.r0 = pos * 2 * BM;
  it.n0 = tile_blocks<CAUSAL>(it.r0, it.len_q, it.len_k);
  it.n1 = tile_blocks<CAUSAL>(it.r0 + BM, it.len_q, it.len_k);
  it.m0 = it.m1 = nullptr;
  it.lim0 = it.lim1 = 0;
  if (SPARSE) {
    const unsigned char* mu = p.bmask + (it.unit / p.H) * p.bm_sb + (it.unit % p.H) * p.bm_sh;
    const int qb = it.r0 / kMaskBlock;
    it.m0 = mu + static_cast<long long>(qb) * p.bm_sq;
    it.m1 = mu + static_cast<long long>(qb + 1) * p.bm_sq;
    // a tile that keeps no block of its range is skipped (its rows are
    // written as empty by the softmax group)
    bool any0 = false, any1 = false;
    for (int j = 0; j < it.n0 && !any0; ++j) any0 = it.m0[j] != 0;
    for (int j = 0; j < it.n1 && !any1; ++j) any1 = it.m1[j] != 0;
    it.lim0 = any0 ? it.n0 : 0;
    it.lim1 = any1 ? it.n1 : 0;
    int c0 = 0, c1 = 0;
    for (int j = 0; j < max(it.lim0, it.lim1); ++j) {
      if (!loaded_block(it, j)) continue;
      c0 += j < it.lim0;
      c1 += j < it.lim1;
    }
    it.n0 = c0;
    it.n1 = c1;
  }
  it.nmax = max(it.n0, it.n1);
  return it;
}

// EXT (dense layout only): 0 plain, 1 block-sparse (p.bmask), 2 additive mask
// (p.amask), 3 dropout (p.dropout), 4 plain on strided tensors (p.strided).
template <int D, typename T, bool CAUSAL, bool PACKED, int EXT>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
fwd_tc_kernel(const Problem p, const __grid_constant__ CUtensorMap tmQ,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmM, unsigned* sched) {
  using C = Cfg<D, EXT>;
  constexpr bool SPARSE = EXT == 1, BIAS = EXT == 2, DROP = EXT == 3, STRIDED = EXT == 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Persistent: CTA b starts with work item b (with per-slot pipelines, slot
  // s with item 2b + s), then claims items dynamically.
  constexpr int kClaim = C::kTileStreams ? 2 : 1;       // claimers per CTA
  constexpr int kItemRows = C::kTileStreams ? BM : 2 * BM;
  const int nper = ((PACKED ? p.max_q : p.Lq) + kItemRows - 1) / kItemRows;   // items per unit
  const int nitems = nper * p.B * p.H;

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sSlots = smem_u32(smem + C::kOffSlots);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], C::kTileStreams ? 1 : C::kMmaWarps);   // the ring's consumers
    }
    for (int i = 0; i < 2 * C::kQBufs; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], C::kStageQ ? 4 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], BM);
      mbar_init(&bars->p_full[t], BM);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_free[t], BM);
    }
    for (int i = 0; i < 2 * kItemQueue; ++i) {
      mbar_init(&bars->item_full[i], 1);
      // one arrival per consuming warp: a softmax group and an MMA warp per
      // slot, or both groups and the MMA warp(s)
      mbar_init(&bars->item_empty[i], C::kTileStreams ? 5 : 8 + C::kMmaWarps);
    }
    mbar_init(&bars->done, C::kMmaWarps);
    for (int w = 0; w < 8; ++w) mbar_init(&bars->mfull[w], 1);
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

  if (warp >= 8) {
   // producer, MMA and idle warps
   regs_dec<kRegsControl>();
   // With per-slot pipelines the control group's fourth warp is slot 1's
   // producer: each producer claims its slot's tiles, publishes them on the
   // slot's queue and loads their Q and K/V into the slot's buffers and ring.
   if (warp == kProducerWarp || (C::kTileStreams && warp == kProducerWarp + 3)) {
    // ------------------------------------------------------------ producer
    const int pr = warp == kProducerWarp ? 0 : 1;   // this thread's slot (ring and queue)
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int fill = 0;             // next position in ring pr (K_0, V_0, K_1, V_1, ... per item)
      int qloads[2] = {0, 0};   // Q loads so far per tile
      bool ok = true;
      int idx = kClaim * blockIdx.x + pr;
      for (int k = 0;; ++k) {
        // publish the item (or the end marker) to the slot's consumers
        const int q = pr * kItemQueue + k % kItemQueue;
        if (k >= kItemQueue && !(ok = mbar_wait(&bars->item_empty[q], (k / kItemQueue - 1) & 1, abort_flag, p.status)))
          break;
        if (!ok || idx >= nitems) idx = -1;
        Item it{};
        if (idx >= 0) it = decode_item<CAUSAL, PACKED, SPARSE, C::kTileStreams>(p, idx, nper, pr);
        bars->item[q] = idx;
        bars->item_n[q] = it.nmax;         // the consumers need not count the kept blocks again
        mbar_arrive(&bars->item_full[q]);
        if (idx < 0) break;
        idx = static_cast<int>(atomicAdd(sched, 1u)) + kClaim * static_cast<int>(gridDim.x);
        if (it.nmax == 0) continue;
        // boxes: packed (column, head, token); dense (column, row, unit), or
        // (column, row, head, batch) through the 4-D maps of strided tensors
        auto load = [&](void* dst, const CUtensorMap* m, uint64_t* bar, int col, int row, int tok0) {
          if constexpr (PACKED) tma_load_3d(dst, m, bar, col, it.h, tok0 + row);
          else if constexpr (STRIDED) tma_load_4d(dst, m, bar, col, row, it.unit % p.H, it.unit / p.H);
          else tma_load_3d(dst, m, bar, col, row, it.unit);
        };
        for (int t = C::kTileStreams ? pr : 0; t < (C::kTileStreams ? pr + 1 : 2) && ok; ++t) {
          if ((t == 0 ? it.n0 : it.n1) == 0) continue;
          // buffer qb of tile t was last used kQBufs loads ago
          const int qb = t * C::kQBufs + qloads[t] % C::kQBufs, use = qloads[t] / C::kQBufs;
          if (use > 0 && !(ok = mbar_wait(&bars->q_empty[qb], (use - 1) & 1, abort_flag, p.status))) break;
          ++qloads[t];
          if (p.debug & kDebugDropQArrive) continue;
          mbar_expect_tx(&bars->q_full[qb], C::kTileBytes);
          const int row = it.r0 + t * BM;
          for (int cb = 0; cb < C::kNBlk; ++cb)
            load(smem + C::kOffQ + qb * C::kTileBytes + cb * C::kColBlkBytes, &tmQ, &bars->q_full[qb], cb * C::kBlk,
                 row, it.tok0);
        }
        // K_jk and V_jk into the next two slots of ring pr
        auto fill_block = [&](int jk) {
          for (int kv = 0; kv < 2; ++kv, ++fill) {
            const int slot = pr * C::kRing + fill % C::kRing;
            const int round = fill / C::kRing;
            if (!SDPA_CHECK(slot >= 0 && slot < C::kSlots, p.status)) {
              ok = false;
              *abort_flag = 1u;
              return;
            }
            if (round > 0 && !(ok = mbar_wait(&bars->empty[slot], (round - 1) & 1, abort_flag, p.status))) return;
            mbar_expect_tx(&bars->full[slot], C::kTileBytes);
            const CUtensorMap* m = kv ? &tmV : &tmK;
            const int row = jk * BN;
            for (int cb = 0; cb < C::kNBlk; ++cb)
              load(smem + C::kOffSlots + slot * C::kTileBytes + cb * C::kColBlkBytes, m, &bars->full[slot],
                   cb * C::kBlk, row, it.tok0k);
          }
        };
        if constexpr (C::kTileStreams) {
          // the key blocks this thread's tile keeps
          const unsigned char* mine = pr == 0 ? it.m0 : it.m1;
          const int lim = pr == 0 ? it.lim0 : it.lim1;
          int jk = -1;
          for (int i = 0; i < (pr == 0 ? it.n0 : it.n1) && ok; ++i) {
            jk = next_kept(mine, lim, jk + 1);
            fill_block(jk);
          }
        } else {
          constexpr bool sparse = SPARSE;
          int jk = -1;             // key block of the current loaded block
          for (int j = 0; j < it.nmax && ok; ++j) {
            jk = sparse ? next_loaded(it, jk + 1) : j;
            fill_block(jk);
          }
        }
      }
      // the last claimer to finish resets this launch's scheduler slot
      if (atomicAdd(sched + 1, 1u) == kClaim * gridDim.x - 1) {
        atomicExch(sched, 0u);
        atomicExch(sched + 1, 0u);
      }
      if (*abort_flag) {
        // Let copies already issued land before the CTA's shared memory is released.
        for (int f = max(0, fill - C::kRing); f < fill; ++f)
          mbar_wait_drain(&bars->full[pr * C::kRing + f % C::kRing], (f / C::kRing) & 1);
        for (int t = 0; t < 2; ++t)
          for (int n = max(0, qloads[t] - C::kQBufs); n < qloads[t]; ++n)
            if (!(p.debug & kDebugDropQArrive))
              mbar_wait_drain(&bars->q_full[t * C::kQBufs + n % C::kQBufs], (n / C::kQBufs) & 1);
      }
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + C::kMmaWarps) {
    // ------------------------------------------------------------ MMA issue
    // Warp w serves Q tiles [t_lo, t_hi); lane 0 issues. Without per-tile
    // streams every MMA warp consumes every K/V fill of the one ring (a slot's
    // empty barrier takes one commit from each); with them warp t reads ring t.
    const int t_lo = C::kMmaWarps == 2 ? warp - kMmaWarp : 0;
    const int t_hi = C::kMmaWarps == 2 ? t_lo + 1 : 2;
    const int ring = C::kTileStreams ? t_lo : 0;      // ring and item queue
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __half>::value ? 0u : 1u;
      constexpr uint32_t idS = idesc_f16(fmt, 0, 0, BM, BN);
      constexpr uint32_t idO = idesc_f16(fmt, 0, 1, BM, D);
      // descriptors of the operand tiles; advancing the start address by `off`
      // bytes adds off >> 4 to the descriptor (the address field cannot carry)
      const uint64_t dQ = smem_desc(sQ, 16, C::kSbo, C::kSw);
      const uint64_t dSlot0K = smem_desc(sSlots, 16, C::kSbo, C::kSw);
      const uint64_t dSlot0V = smem_desc(sSlots, C::kColBlkBytes, C::kSbo, C::kSw);
      auto issue_qk = [&](int t, int qb, int slot) {
        const uint64_t a = dQ + ((qb * C::kTileBytes) >> 4);
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
      auto slot_of = [&](int pos) { return ring * C::kRing + pos % C::kRing; };
      auto full_wait = [&](int pos) { return wait(&bars->full[slot_of(pos)], (pos / C::kRing) & 1); };
      // Work items come from the producer's queue; the next one is read ahead
      // so that its first S_t can be issued before the current item's last P.V.
      int k = 0;                 // queue index of the current item
      int next_idx = -2;         // queue entry k + 1 once read (-2: not yet)
      int kept = -1;             // the current item's kept blocks (per-slot pipelines)
      auto take = [&](int kk, int& idx) {
        const int q = ring * kItemQueue + kk % kItemQueue;
        if (!wait(&bars->item_full[q], (kk / kItemQueue) & 1)) return false;
        idx = *reinterpret_cast<volatile int*>(&bars->item[q]);
        if (C::kTileStreams) kept = *reinterpret_cast<volatile int*>(&bars->item_n[q]);
        mbar_arrive(&bars->item_empty[q]);
        return true;
      };
      int fill = 0;              // position of the current item's K_0 in this warp's ring
      int qloads[2] = {0, 0};    // Q tiles consumed per tile slot
      int blocks[2] = {0, 0};    // K/V blocks processed per tile slot (barrier phases)
      int items[2] = {0, 0};     // work items finished per tile slot
      bool pre[2] = {false, false};   // first S_t of the current item already issued
      // first S_t = Q_t K_0^T of item `x` whose K_0 sits at ring position `xfill`
      auto first_qk = [&](const Item& x, int t, int xfill) {
        const int nt = t == 0 ? x.n0 : x.n1;
        const int qb = t * C::kQBufs + qloads[t] % C::kQBufs;
        if (!wait(&bars->q_full[qb], (qloads[t] / C::kQBufs) & 1)) return false;
        ++qloads[t];
        // the tile's previous S_t must have been read (P overlaying S is
        // ordered behind the last P.V on the tensor cores instead)
        if (!C::kPAlias && blocks[t] > 0 && !wait(&bars->s_free[t], (blocks[t] - 1) & 1)) return false;
        if (!full_wait(xfill)) return false;
        tc_fence_after();
        issue_qk(t, qb, slot_of(xfill));
        mma_commit(&bars->s_full[t]);
        if (!C::kStageQ && nt == 1) mma_commit(&bars->q_empty[qb]);
        return true;
      };
      bool ok = true;
      int idx = -1;
      ok = take(0, idx);
      while (ok && idx >= 0) {
        const Item it = decode_item<CAUSAL, PACKED, SPARSE, C::kTileStreams>(p, idx, nper, t_lo, kept);
        int qbuf[2];             // Q buffer of this item per tile
        for (int t = t_lo; t < t_hi; ++t) qbuf[t] = t * C::kQBufs + (qloads[t] - (pre[t] ? 1 : 0)) % C::kQBufs;
        if (it.nmax > 0) {
          for (int t = t_lo; t < t_hi && ok; ++t) {
            if ((t == 0 ? it.n0 : it.n1) == 0 || pre[t]) continue;
            qbuf[t] = t * C::kQBufs + qloads[t] % C::kQBufs;
            // With an MMA warp per tile, tile 1 starts the CTA's first item
            // once tile 0 has handed over its first P, so the two softmax
            // groups run about half a block apart from then on: one group's
            // TMEM loads and waits fall under the other's exponentials
            // instead of both groups loading, then competing for the
            // exponential unit, at the same moments.
            if (C::kMmaWarps == 2 && !C::kTileStreams && t == 1 && k == 0 && it.n0 > 0 &&
                !(ok = wait(&bars->p_full[0], 0)))
              break;
            ok = first_qk(it, t, fill);
          }
          if (!ok) break;
          if (item_fills(it, C::kTileStreams, ring) > 0) mma_commit(&bars->empty[slot_of(fill)]);   // K_0 consumed
        }
        pre[0] = pre[1] = false;   // from here on pre[] is about the next item
        // blocks this warp walks: the item's loaded blocks, or with per-tile
        // streams its own tile's kept blocks
        const int jmax = item_fills(it, C::kTileStreams, ring) / 2;
        for (int j = 0; j < jmax && ok; ++j) {
          // K_{j+1} sits at ring position fill + 2j + 2, V_j at fill + 2j + 1
          const bool has_next = j + 1 < jmax;
          const int kpos = fill + 2 * j + 2;
          const int vpos = fill + 2 * j + 1;
          if (has_next && !(ok = full_wait(kpos))) break;
          if (!(ok = full_wait(vpos))) break;
          tc_fence_after();
          for (int t = t_lo; t < t_hi && ok; ++t) {
            const int nt = t == 0 ? it.n0 : it.n1;
            if (j >= nt) continue;
            const int g = blocks[t] + j;
            if (!C::kPAlias && j + 1 < nt) {
              // S_t may be overwritten once its softmax group holds it in registers
              if (!(ok = wait(&bars->s_free[t], g & 1))) break;
              tc_fence_after();
              issue_qk(t, qbuf[t], slot_of(kpos));
              mma_commit(&bars->s_full[t]);
              if (!C::kStageQ && j + 2 == nt) mma_commit(&bars->q_empty[qbuf[t]]);
            } else if (!C::kPAlias && !C::kTileStreams && j + 1 == nt) {
              // last block of this tile: read the next work item and issue its
              // first S_t now, under this block's softmax
              if (next_idx == -2 && !(ok = take(k + 1, next_idx))) break;
              if (next_idx >= 0) {
                const Item nx = decode_item<CAUSAL, PACKED, SPARSE, C::kTileStreams>(p, next_idx, nper, t_lo);
                if (nx.nmax > 0 && (t == 0 ? nx.n0 : nx.n1) > 0) {
                  blocks[t] += nt;            // the phases of S_t continue into the next item
                  ok = first_qk(nx, t, fill + item_fills(it, C::kTileStreams, ring));
                  blocks[t] -= nt;
                  if (!ok) break;
                  pre[t] = true;
                }
              }
            }
            if (!(ok = wait(&bars->p_full[t], g & 1))) break;
            // O_t is overwritten by the item's first P.V: the previous item's
            // epilogue must have read it
            if (j == 0 && items[t] > 0 && !(ok = wait(&bars->o_free[t], (items[t] - 1) & 1))) break;
            tc_fence_after();
            issue_pv(t, slot_of(vpos), j > 0);
            mma_commit(&bars->pv_done[t]);
            if (C::kPAlias && j + 1 < nt) {
              // P_t overlays S_t: the next S_t is issued behind the MMA that reads P_t
              issue_qk(t, qbuf[t], slot_of(kpos));
              mma_commit(&bars->s_full[t]);
              if (!C::kStageQ && j + 2 == nt) mma_commit(&bars->q_empty[qbuf[t]]);
            }
          }
          mma_commit(&bars->empty[slot_of(vpos)]);
          if (has_next) mma_commit(&bars->empty[slot_of(kpos)]);
        }
        if (!ok) break;
        for (int t = t_lo; t < t_hi; ++t) {
          const int nt = t == 0 ? it.n0 : it.n1;
          blocks[t] += nt;
          if (nt > 0) ++items[t];
        }
        fill += item_fills(it, C::kTileStreams, ring);
        ++k;
        if (next_idx != -2) {
          idx = next_idx;
          next_idx = -2;
        } else {
          ok = take(k, idx);
        }
      }
      mma_commit(&bars->done);
      mbar_wait_drain(&bars->done, 0);
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = warp / 4;
    const int rl = threadIdx.x & 127;        // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS + t * BN;
    const uint32_t tO = tmem + lane_off + C::kColO + t * D;
    const uint32_t tP = tmem + lane_off + C::kColP + t * C::kPStride;
    const float c = p.scale * kLog2e;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      // warp-uniform decision: the TMEM accesses that follow are warp-collective
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
    };
    int blocks = 0;   // K/V blocks processed by this tile slot so far (barrier phases)
    // Epilogue of a finished work item: O = O / l rounded once, LSE = (m + log2 l) ln 2.
    // Where a CTA runs many items (d <= 64) it is deferred into the next item's
    // first block, after that block's P has been handed to the tensor cores, so
    // the wait for the item's last P.V overlaps the next item's exponentials.
    constexpr bool kDefer = !C::kPAlias;
    struct Pending {
      bool on;
      float m, l;
      long long orow, li;     // output row offset (elements) and LSE index; orow < 0: row past the end
      int qb;                 // the item's Q buffer
    } pend{false, 0.f, 0.f, -1, 0, 0};
    int qn = 0;               // Q tiles this group's tile has been loaded with
    auto epilogue = [&](const Pending& e) {
      tc_fence_after();
      // l = 0 only for a row with no visible key (block-sparse): O = 0, LSE = -inf
      const float inv = e.l > 0.f ? __frcp_rn(e.l) : 0.f;
      uint32_t ov[D / 2];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          ov[cc * 16 + x] = Pack2<T>::pack(__uint_as_float(o[2 * x]) * inv, __uint_as_float(o[2 * x + 1]) * inv);
      }
      // O_t has been read out: the next item's first P.V may overwrite it
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
      if constexpr (C::kStageQ || C::kStageO) {
        // The warp's 32 rows go through shared memory: each lane writes its
        // row as 16-byte chunks (chunk c of row r at slot c ^ f(r), so the 8
        // lanes of a quarter-warp hit 8 different bank groups), then each
        // store instruction takes whole rows, 512 contiguous bytes of them
        // where rows are adjacent, instead of 32 rows of 16 bytes each.
        constexpr int kChunks = D / 8;                     // 16-byte chunks per row
        constexpr int kRowsPer = 32 / kChunks;             // rows per store instruction
        auto slot = [](int r, int c) { return c ^ (kChunks == 8 ? (r & 7) : ((r >> 1) & 3)); };
        // the staging Q buffer must be one of this tile's (else, in the debug
        // build, the tile's first one: the status word already says the
        // output is invalid)
        const int qb = SDPA_CHECK(!C::kStageQ || (e.qb >= t * C::kQBufs && e.qb < (t + 1) * C::kQBufs), p.status)
                           ? e.qb
                           : t * C::kQBufs;
        const uint32_t stage = C::kStageQ
                                   ? smem_u32(smem + C::kOffQ + qb * C::kTileBytes + (warp & 3) * C::kStageWarpBytes)
                                   : smem_u32(smem + C::kOffStage + warp * C::kStageWarpBytes);
        if (C::kStageO) __syncwarp();                      // the previous epilogue's reads are done
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       ::"r"(stage + (lane * kChunks + slot(lane, c)) * 16), "r"(ov[4 * c]), "r"(ov[4 * c + 1]),
                         "r"(ov[4 * c + 2]), "r"(ov[4 * c + 3]) : "memory");
        __syncwarp();
        const int c = lane % kChunks;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
          const int r = i * kRowsPer + lane / kChunks;     // the row this lane stores a chunk of
          const long long orow = __shfl_sync(0xffffffffu, e.orow, r);
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w) : "r"(stage + (r * kChunks + slot(r, c)) * 16)
                       : "memory");
          if (orow >= 0 && SDPA_CHECK(orow + 8 * c + 8 <= p.ext[kTo], p.status))
            *reinterpret_cast<uint4*>(static_cast<T*>(p.o) + orow + 8 * c) = w;
        }
        if constexpr (C::kStageQ) {
          // the staged rows have been read out: the producer may load the next
          // Q into the buffer (its copy is an async-proxy write after these
          // generic accesses)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->q_empty[qb]);
        }
        if (e.orow >= 0 && SDPA_CHECK(e.li < p.lse_ext, p.status))
          p.lse[e.li] = e.l > 0.f ? (e.m + __log2f(e.l)) * kLn2 : -INFINITY;
      } else if (e.orow >= 0 && SDPA_CHECK(e.orow + D <= p.ext[kTo] && e.li < p.lse_ext, p.status)) {
        T* orow = static_cast<T*>(p.o) + e.orow;
#pragma unroll
        for (int x = 0; x < D / 8; ++x)
          *reinterpret_cast<uint4*>(orow + 8 * x) = make_uint4(ov[4 * x], ov[4 * x + 1], ov[4 * x + 2], ov[4 * x + 3]);
        p.lse[e.li] = e.l > 0.f ? (e.m + __log2f(e.l)) * kLn2 : -INFINITY;
      }
    };
    // Additive mask: each warp loads its own 32 rows x BN keys of a block
    // with TMA into its slot (mcons loads consumed, missued issued so far).
    int mcons = 0, missued = 0;
    auto issue_mask = [&](const Item& x, int kb) {
      // the slot's previous contents have been read by every lane
      __syncwarp();
      fence_proxy_async_smem();
      if (lane == 0) {
        uint8_t* dst = smem + C::kOffMask + warp * C::kMaskWarpBytes;
        const int zc = p.am_sh ? x.unit % p.H : 0, wc = p.am_sb ? x.unit / p.H : 0;
        const int r0w = x.r0 + t * BM + (warp & 3) * 32;     // this warp's first row within the unit
        mbar_expect_tx(&bars->mfull[warp], C::kMaskWarpBytes);
        for (int h = 0; h < 2; ++h)
          tma_load_4d(dst + h * (C::kMaskWarpBytes / 2), &tmM, &bars->mfull[warp], kb + h * (BN / 2), r0w, zc, wc);
      }
      ++missued;
    };
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int q = (C::kTileStreams ? t * kItemQueue : 0) + k % kItemQueue;
      if (!(ok = wait_all(&bars->item_full[q], (k / kItemQueue) & 1))) break;
      const int idx = *reinterpret_cast<volatile int*>(&bars->item[q]);
      const int kept = C::kTileStreams ? *reinterpret_cast<volatile int*>(&bars->item_n[q]) : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[q]);
      if (idx < 0) break;
      const Item it = decode_item<CAUSAL, PACKED, SPARSE, C::kTileStreams>(p, idx, nper, t, kept);
      const int nt = t == 0 ? it.n0 : it.n1;
      const int rt = it.r0 + t * BM;
      const int row = rt + rl;                // row within the unit
      if (nt == 0) {
        // block-sparse: a tile whose mask row keeps nothing has no visible key:
        // O = 0, LSE = -inf
        const long long ro = (static_cast<long long>(it.unit) * it.len_q + row) * D;
        if (SPARSE && row < it.len_q && SDPA_CHECK(ro + D <= p.ext[kTo] && ro / D < p.lse_ext, p.status)) {
          T* orow = static_cast<T*>(p.o) + ro;
#pragma unroll
          for (int x = 0; x < D / 8; ++x) *reinterpret_cast<uint4*>(orow + 8 * x) = make_uint4(0u, 0u, 0u, 0u);
          p.lse[static_cast<long long>(it.unit) * it.len_q + row] = -INFINITY;
        }
        continue;
      }
      const int qb_item = t * C::kQBufs + qn % C::kQBufs;   // the producer loaded this tile's Q there
      ++qn;
      constexpr bool sparse = SPARSE;
      const unsigned char* mine = t == 0 ? it.m0 : it.m1;
      if (BIAS) issue_mask(it, 0);           // the item's first mask block
      int jk = -1;                           // key block of the current loaded block
      float m_run = -INFINITY, l = 0.f;      // maximum used in the exponent (base 2), running sum
      for (int j = 0; j < nt; ++j) {
        const int g = blocks + j;
        jk = !sparse ? j : C::kTileStreams ? next_kept(mine, t == 0 ? it.lim0 : it.lim1, jk + 1)
                                           : next_loaded(it, jk + 1);
        const int kbase = jk * BN;
        if (sparse && !mine[jk]) {
          // A loaded block this tile's mask row drops: its probabilities are
          // all 0, so P_t = 0 goes to the tensor cores with the same handshakes
          // as any block, and the max, exponentials and rescale are skipped.
          if (!(ok = wait_all(&bars->s_full[t], g & 1))) break;
          if (!C::kPAlias) {
            tc_fence_before();
            mbar_arrive(&bars->s_free[t]);
          }
          // P_t's columns are free once the previous P.V on this tile has finished
          if (!C::kPAlias && (j > 0 || pend.on) && !(ok = wait_all(&bars->pv_done[t], (g - 1) & 1))) break;
          tc_fence_after();
          uint32_t zero[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) zero[i] = 0u;
          tmem_st32(tP, zero);
          tmem_st32(tP + 32, zero);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full[t]);
          if (kDefer && j == 0 && pend.on) {
            epilogue(pend);
            pend.on = false;
          }
          continue;
        }
        // additive mask: this row's BN entries from the warp's slot (two
        // 64-key boxes, 128-byte swizzled: 16-byte chunk c of row r sits at
        // chunk c ^ (r % 8)); once read, the slot takes the next block's mask,
        // which lands while this block computes
        uint4 am[BIAS ? BN / 8 : 1];
        if (BIAS) {
          if (!(ok = wait_all(&bars->mfull[warp], mcons & 1))) break;
          ++mcons;
          const uint8_t* ms = smem + C::kOffMask + warp * C::kMaskWarpBytes + lane * 128;
#pragma unroll
          for (int u = 0; u < BN / 8; ++u)
            am[u] = *reinterpret_cast<const uint4*>(ms + (u / 8) * (C::kMaskWarpBytes / 2) + (((u % 8) ^ (lane & 7)) << 4));
          if (j + 1 < nt) issue_mask(it, kbase + BN);
        }
        if (!(ok = wait_all(&bars->s_full[t], g & 1))) break;
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
        if (BIAS) {
          // x = S * scale + M, the exponent in natural-log units; the max and
          // the exponentials below scale it by log2(e) like they scale S by
          // scale * log2(e) without a mask
#pragma unroll
          for (int u = 0; u < BN / 8; ++u) {
            const uint32_t w[4] = {am[u].x, am[u].y, am[u].z, am[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 mf = Pack2<T>::unpack(w[e]);
              x[8 * u + 2 * e] = fmaf(x[8 * u + 2 * e], p.scale, mf.x);
              x[8 * u + 2 * e + 1] = fmaf(x[8 * u + 2 * e + 1], p.scale, mf.y);
            }
          }
        }
        if ((kbase + BN > it.len_k) || (CAUSAL && kbase + BN - 1 > rt)) {
          // keys kbase + i with i >= lim are past the end or (causal) after the row
          const int lim = (CAUSAL ? min(it.len_k, row + 1) : it.len_k) - kbase;
#pragma unroll
          for (int i = 0; i < BN; ++i) x[i] = i < lim ? x[i] : -INFINITY;
        }
        // exponentials of one half of the block (BN / 2 keys) against the
        // exponent offset mu, packed for TMEM; the sums keep every probability
        auto exps_half = [&](int half, float mu, uint32_t (&pk)[BN / 4], float& s0, float& s1, float& s2,
                             float& s3) {
          uint4 rnd = make_uint4(0u, 0u, 0u, 0u);   // dropout bytes of the current 16 keys
#pragma unroll
          for (int chunk = 0; chunk < BN / 16; ++chunk) {
            const float* xc = x + half * (BN / 2) + chunk * 8;
            float e[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              fma2(e[2 * u], e[2 * u + 1], xc[2 * u], xc[2 * u + 1], BIAS ? kLog2e : c, -mu);
              e[2 * u] = ex2_approx(e[2 * u]);
              e[2 * u + 1] = ex2_approx(e[2 * u + 1]);
            }
            add2(s0, s1, e[0], e[1]);
            add2(s2, s3, e[2], e[3]);
            add2(s0, s1, e[4], e[5]);
            add2(s2, s3, e[6], e[7]);
            if (DROP) {
              // the row sum above keeps every probability; P . V sees the
              // dropped and rescaled ones
              if ((chunk & 1) == 0)
                rnd = philox4x32_10(make_uint4(static_cast<uint32_t>(jk * (BN / 16) + half * (BN / 32) + chunk / 2),
                                               static_cast<uint32_t>(row), static_cast<uint32_t>(it.unit), 0u),
                                    p.seed_lo, p.seed_hi);
              const uint32_t w0 = (chunk & 1) ? rnd.z : rnd.x, w1 = (chunk & 1) ? rnd.w : rnd.y;
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const uint32_t byte = ((u < 4 ? w0 : w1) >> (8 * (u & 3))) & 0xffu;
                e[u] = byte >= p.drop_t ? e[u] * p.drop_scale : 0.f;
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) pk[chunk * 4 + u] = Pack2<T>::pack(e[2 * u], e[2 * u + 1]);
          }
        };
        // P_t's columns are free once the previous P.V on this tile (possibly
        // the last one of the previous item) has finished; at d = 128 they
        // overlay S_t, already in registers, and that MMA finished before S_j
        bool waited = C::kPAlias || !(j > 0 || pend.on);
        auto wait_p_free = [&]() {
          if (!waited) ok = wait_all(&bars->pv_done[t], (g - 1) & 1);
          waited = true;
        };
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        bool grow = false;
        float m_new = m_run, alpha = 1.f;
        bool done = false;
        if (D == 128 && j > 0) {
          // After the first block the running maximum is usually still good
          // enough: exponentiate against it and keep the result if the block's
          // probabilities sum to at most 2^kRescaleThreshold (so each is at most
          // that, the bound the lazy rescale allows). Otherwise fall back to
          // the block's own maximum below. Softmax is shift invariant, so both
          // give the same result; the first avoids the max pass. (Measured: it
          // pays at d = 128; at d <= 64 the extra warp votes cost more.)
          const float mu = m_run == -INFINITY ? 0.f : m_run;
          constexpr float kSumLimit = 256.f;   // 2^kRescaleThreshold
          uint32_t pk[BN / 4];
          exps_half(0, mu, pk, s0, s1, s2, s3);
          if (!__any_sync(0xffffffffu, (s0 + s1) + (s2 + s3) > kSumLimit)) {
            wait_p_free();
            if (!ok) break;
            tmem_st32(tP, pk);
            float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
            exps_half(1, mu, pk, t0, t1, t2, t3);
            const float tot = ((s0 + s1) + (s2 + s3)) + ((t0 + t1) + (t2 + t3));
            if (!__any_sync(0xffffffffu, tot > kSumLimit)) {
              tmem_st32(tP + 32, pk);
              s0 += t0;
              s1 += t1;
              s2 += t2;
              s3 += t3;
              // the offset used becomes the running maximum (it differs only
              // for a row whose earlier keys were all masked: then l = 0, O = 0)
              m_new = mu;
              alpha = ex2_approx(m_run - mu);
              done = true;
            }
          }
        }
        if (!done) {
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
          const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3)) * (BIAS ? kLog2e : c);
          grow = mx > m_run + kRescaleThreshold;
          m_new = grow ? mx : m_run;
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          alpha = ex2_approx(m_run - m_use);
          // exponentials into packed registers, stored to TMEM in two halves; the
          // first half is computed before waiting for P_t's columns to be free
          s0 = s1 = s2 = s3 = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[BN / 4];
            exps_half(half, m_use, pk, s0, s1, s2, s3);
            if (half == 0) wait_p_free();
            if (!ok) break;
            tmem_st32(tP + half * 32, pk);
          }
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
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
        if (kDefer && j == 0 && pend.on) {
          // the previous item's last P.V was waited for above
          epilogue(pend);
          pend.on = false;
        }
      }
      if (!ok) break;
      blocks += nt;
      pend.on = true;
      pend.m = m_run;
      pend.l = l;
      pend.qb = qb_item;
      pend.orow = row < it.len_q ? (PACKED    ? (static_cast<long long>(it.tok0 + row) * p.H + it.h) * D
                                    : STRIDED ? dense_off(p, kTo, it.unit / p.H, it.unit % p.H, row)
                                              : (static_cast<long long>(it.unit) * it.len_q + row) * D)
                                 : -1;
      pend.li = PACKED ? static_cast<long long>(it.h) * p.Lq + it.tok0 + row
                       : static_cast<long long>(it.unit) * it.len_q + row;
      if (!kDefer) {
        if (!(ok = wait_all(&bars->pv_done[t], (blocks - 1) & 1))) break;
        epilogue(pend);
        pend.on = false;
      }
    }
    if (ok && pend.on && wait_all(&bars->pv_done[t], (blocks - 1) & 1)) epilogue(pend);
    // after a failed wait, let a mask load still in flight land before the
    // CTA's shared memory is released
    if (BIAS && missued > mcons && lane == 0) mbar_wait_drain(&bars->mfull[warp], mcons & 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
  }
}

template <int D, typename T, bool CAUSAL, bool PACKED, int EXT>
cudaError_t launch_one(const Problem& p, const FwdMaps& m, cudaStream_t s) {
  auto kern = fwd_tc_kernel<D, T, CAUSAL, PACKED, EXT>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, EXT>::kSmem);
    if (e != cudaSuccess) return e;
    // setmaxnreg redistributes the registers the block is launched with; a
    // split larger than that would wait forever, so refuse to launch instead
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * Cfg<D>::kThreads < static_cast<int>(256 * kRegsSoftmax + 128 * kRegsControl)) return cudaErrorInvalidConfiguration;
    attr_set[dev] = 1;
  }
  static int sm_count[64] = {0};
  if (dev < 64 && sm_count[dev] == 0) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int sms = dev < 64 ? sm_count[dev] : 1;
  const int rows = PACKED ? p.max_q : p.Lq;
  constexpr bool kTiles = Cfg<D, EXT>::kTileStreams;     // two single-tile claimers per CTA
  const long long nper = (rows + (kTiles ? BM : 2 * BM) - 1) / (kTiles ? BM : 2 * BM);
  const long long items = nper * p.B * p.H;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // d <= 64: persistent, one CTA per SM (each needs most of the SM's SMEM and all
  // of its TMEM) claiming items until none are left, so an item's prologue and
  // epilogue overlap its neighbours'. d = 128: one CTA per item measured faster
  // (its items are long, and the hardware's block scheduler balances them).
  const long long ctas = kTiles ? (items + 1) / 2 : items;
  const long long want = D == 128 ? items : (ctas < sms ? ctas : sms);
  const unsigned grid = static_cast<unsigned>(want);
  static unsigned* sched_base[64] = {nullptr};
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (sched_base[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_fwd_sched);
    if (e != cudaSuccess) return e;
    sched_base[dev] = static_cast<unsigned*>(ptr);
  }
  static std::atomic<unsigned> launches{0};
  unsigned* sched = sched_base[dev] + 2 * (launches.fetch_add(1) % kSchedSlots);
  kern<<<grid, Cfg<D>::kThreads, Cfg<D, EXT>::kSmem, s>>>(p, m.q, m.k, m.v, m.mask, sched);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_d(const Problem& p, const FwdMaps& m, cudaStream_t s) {
  const bool packed = p.cu_seqlens != nullptr;
  if (p.bmask != nullptr)
    return p.causal ? launch_one<D, T, true, false, 1>(p, m, s) : launch_one<D, T, false, false, 1>(p, m, s);
  if (p.amask != nullptr)
    return p.causal ? launch_one<D, T, true, false, 2>(p, m, s) : launch_one<D, T, false, false, 2>(p, m, s);
  if (p.dropout)
    return p.causal ? launch_one<D, T, true, false, 3>(p, m, s) : launch_one<D, T, false, false, 3>(p, m, s);
  if (p.strided)
    return p.causal ? launch_one<D, T, true, false, 4>(p, m, s) : launch_one<D, T, false, false, 4>(p, m, s);
  if (p.causal)
    return packed ? launch_one<D, T, true, true, 0>(p, m, s) : launch_one<D, T, true, false, 0>(p, m, s);
  return packed ? launch_one<D, T, false, true, 0>(p, m, s) : launch_one<D, T, false, false, 0>(p, m, s);
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
