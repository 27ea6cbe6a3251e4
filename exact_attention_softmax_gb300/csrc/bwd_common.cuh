// bwd_common.cuh -- definitions shared by the tensor-core backward kernels
// (bwd_tc.cu: one CTA per 128-key block; bwd_persist.cu: persistent CTAs
// that claim key blocks): warp roles, the shared-memory and TMEM plan, the
// barrier block and small device helpers (internal).
#pragma once

#include <type_traits>

#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int BK = 128;          // keys per CTA
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaSWarp = 13;
constexpr int kMmaGWarp = 14;
constexpr int kMaskWarp = 15;    // additive mask loads (the warp idles otherwise)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
// Register split (launch: 512 threads x 128): softmax groups 160, dQ drain and
// control groups 96; 256 * 160 + 256 * 96 = 65536 = 512 * 128, and per SM
// sub-partition 160 + 160 + 96 + 96 = 512 registers per lane.
constexpr uint32_t kRegsSoftmax = 160;
constexpr uint32_t kRegsOther = 96;

template <int D, int EXT>
struct BCfg {
  static constexpr int BQ = D == 128 ? 64 : 128;            // query rows per step
  static constexpr int kHalf = BQ / 2;                       // query columns per softmax group
  static constexpr bool kDqT = D == 128;                     // dQ computed transposed
  // Which MMA warp issues the dQ MMAs, so the two warps issue about as many
  // MMAs per tile: d <= 64 -> the S^T/dP^T warp (d = 64: 8 + 8 vs 16, d = 32:
  // 4 + 8 vs 16), d = 128 -> the dV/dK warp (16 vs 8 + 8).
  static constexpr bool kDqOnS = D <= 64;
  static constexpr int kBlk = D >= 64 ? 64 : D;
  static constexpr int kNBlk = D / kBlk;
  static constexpr uint32_t kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kRowBytes = kBlk * 2;
  static constexpr int kSbo = 8 * kRowBytes;
  static constexpr int kKColBlk = BK * kRowBytes;            // column block of a K/V tile
  static constexpr int kQColBlk = BQ * kRowBytes;            // column block of a Q/dO tile
  static constexpr int kKTile = BK * D * 2;
  static constexpr int kQTile = BQ * D * 2;
  static constexpr int kPColBlk = BK * 128;                  // P^T / dS^T: [128 keys][64 queries] blocks
  static constexpr int kPBytes = BK * BQ * 2;
  // Q/dO stages: a stage stays busy from its load until the dV/dK MMAs of
  // its step, about one step after its S^T MMA; a third stage lets the next
  // load start early enough at d <= 64 (the additive-mask kernel, with its
  // mask ring, has no room for it; at d = 128, with dS^T in TMEM, a third
  // stage measured slower: 5140 against 5091 us on the long causal batch)
  static constexpr bool kMask = EXT == 2;
  static constexpr int kStages = D <= 64 && !kMask ? 3 : 2;
  // shared memory map
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKTile;
  static constexpr int kOffQ = kOffV + kKTile;                          // kStages Q tiles
  static constexpr int kOffDO = kOffQ + kStages * kQTile;               // kStages dO tiles
  static constexpr int kOffDST = kOffDO + kStages * kQTile;            // dS^T (P^T lives in TMEM)
  static constexpr int kDqBytes = kDqT ? BQ * D * 4 : 0;     // fp32 dQ staging tile (d = 128 only)
  static constexpr int kOffDQ = kOffDST + kPBytes;
  static constexpr int kOffStat = kOffDQ + kDqBytes;                    // kStages x (lse2[BQ], delta[BQ])
  // block-sparse: the CTA's active query steps (uint16 indices); additive
  // mask: a ring of two slots, each 32 query rows x 128 keys for both
  // softmax groups (the same region)
  static constexpr int kMaxSteps = 2048;
  static constexpr int kMaskTile = 32 * BK * 2;
  static constexpr int kMaskSlot = 2 * kMaskTile;
  // d = 64: each dQ drain warp stages 32 rows x 32 columns of fp32 (4 KB)
  // so its reductions go out as whole row segments
  static constexpr int kDqStageBytes = kDqT ? 0 : 4 * 32 * 32 * 4;
  static constexpr int kOffDqStage = kOffStat + kStages * BQ * 8;
  static constexpr int kOffList = kOffDqStage + kDqStageBytes;
  static constexpr int kOffBar = kOffList + (kMask ? 2 * kMaskSlot : kMaxSteps * 2);
  static constexpr int kSmem = kOffBar + 256 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
  // TMEM columns: S^T, dP^T, dV, dK, one dQ buffer (its drain takes well
  // under a step), and P^T (BQ 16-bit values per key row, two per column),
  // which the dV MMA reads as its A operand, so P^T costs no shared memory
  static constexpr int kDqCols = kDqT ? BQ : D;
  static constexpr uint32_t kTS = 0, kTdP = BQ, kTdV = 2 * BQ, kTdK = 2 * BQ + D, kTdQ = 2 * BQ + 2 * D;
  static constexpr uint32_t kTP = kTdQ + kDqCols;
  // d = 128 has room for dS^T as well (the dK MMA's A operand; dS^T still
  // goes to shared memory, where the dQ MMA reads it)
  static constexpr bool kDsTmem = D == 128;
  static constexpr uint32_t kTDS = kTP + BQ / 2;
  static_assert(kTP + BQ / 2 + (kDsTmem ? BQ / 2 : 0) <= 512, "TMEM budget");
  static_assert(kStages <= 3, "the barrier arrays hold 3 Q/dO stages");
};

struct __align__(8) BBars {
  uint64_t kv;
  uint64_t full[3];
  uint64_t empty[3];
  uint64_t s_full;     // S^T of the current tile in TMEM
  uint64_t dp_full;    // dP^T of the current tile in TMEM
  uint64_t s_free;     // S^T and dP^T read into registers by both softmax groups
  uint64_t pds_full;   // P^T, dS^T in TMEM / shared memory (d = 128: dS^T only)
  uint64_t pds_free;   // ... consumed by the dV, dK, dQ MMAs (d = 128: dK, dQ)
  uint64_t p_full;     // d = 128: P^T in TMEM, ahead of dS^T
  uint64_t p_free;     // ... consumed by the dV MMAs
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t kv_done;
  uint64_t done;
  uint64_t mfull[2];   // additive mask slot loaded
  uint64_t mempty[2];  // ... read by the 8 softmax warps
  uint32_t tmem_base;
  uint32_t abort_flag;
  int nsteps;          // block-sparse: number of active query steps
};
static_assert(sizeof(BBars) <= 256, "the barrier block has 256 bytes of shared memory");

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
               ::"l"(gdst), "r"(ssrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void red_add_v4_f32(float* gdst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gdst), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16 x 16 byte transpose across the half-warp that holds lanes hl = 0..15:
// on entry byte k of lane hl's 16 bytes belongs to lane k, on return byte c
// of lane k's 16 bytes came from lane c. Four butterfly stages; stage j
// swaps bit j of the lane index with bit j of the byte index, exchanging 8
// of the 16 bytes with lane hl ^ 2^j (two shuffles a stage).
__device__ __forceinline__ void transpose16_bytes(uint32_t (&w)[4], int hl) {
  {
    const bool b = hl & 8;
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, b ? w[0] : w[2], 8);
    const uint32_t rb = __shfl_xor_sync(0xffffffffu, b ? w[1] : w[3], 8);
    if (b) { w[0] = ra; w[1] = rb; } else { w[2] = ra; w[3] = rb; }
  }
  {
    const bool b = hl & 4;
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, b ? w[0] : w[1], 4);
    const uint32_t rb = __shfl_xor_sync(0xffffffffu, b ? w[2] : w[3], 4);
    if (b) { w[0] = ra; w[2] = rb; } else { w[1] = ra; w[3] = rb; }
  }
  // bytes within a word: send the half (then byte) the partner owns, keep the
  // rest, and put the partner's bytes where the sent ones were
  {
    const bool b = hl & 2;
    const uint32_t sel = b ? 0x5410u : 0x7632u, p0 = b ? 0x3254u : 0x5410u, p1 = b ? 0x3276u : 0x7610u;
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, __byte_perm(w[0], w[1], sel), 2);
    const uint32_t rb = __shfl_xor_sync(0xffffffffu, __byte_perm(w[2], w[3], sel), 2);
    w[0] = __byte_perm(w[0], ra, p0); w[1] = __byte_perm(w[1], ra, p1);
    w[2] = __byte_perm(w[2], rb, p0); w[3] = __byte_perm(w[3], rb, p1);
  }
  {
    const bool b = hl & 1;
    const uint32_t sel = b ? 0x6420u : 0x7531u, p0 = b ? 0x3514u : 0x5240u, p1 = b ? 0x3716u : 0x7260u;
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, __byte_perm(w[0], w[1], sel), 1);
    const uint32_t rb = __shfl_xor_sync(0xffffffffu, __byte_perm(w[2], w[3], sel), 1);
    w[0] = __byte_perm(w[0], ra, p0); w[1] = __byte_perm(w[1], ra, p1);
    w[2] = __byte_perm(w[2], rb, p0); w[3] = __byte_perm(w[3], rb, p1);
  }
}

}  // namespace

// Persistent backward (d <= 64, plain and strided tensors, dense or packed),
// in bwd_persist.cu.
template <int D, typename T>
cudaError_t launch_bwd_persist(const BwdProblem& bp, const BwdMaps& m, cudaStream_t s);

}  // namespace sdpa
