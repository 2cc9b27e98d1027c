// attn_fwd_kernel.cuh - fused, tiled attention forward for sm_103a (tcgen05 + TMA).
//
// What is computed (FlashAttention（V3）深度解析, dtcms.com, sections 2, 4.2, 11):
//   S = scale * Q K^T (+ causal mask: key j visible to query i iff j <= i),
//   P = softmax(S) row-wise, O = P V, LSE = ln sum_j exp(S_ij),
// with S and P never leaving the SM: each 128-key block of K/V is streamed
// through shared memory and folded into a running FP32 (max, sum, O) per query
// row with the merge rule m = max(m_a, m_b), z = z_a e^(m_a-m) + z_b e^(m_b-m)
// (section 4.2).
//
// Blackwell mapping (the pages' Hopper design - TMA producer warps, WGMMA
// consumers, inter-warpgroup ping-pong, section 7.3 - redone for tcgen05):
//   * one persistent CTA per SM walks work units (b, query head, block of
//     QST x 128 query rows); QST = 2 query tiles share every K/V tile;
//   * load warp: one thread issues TMA copies of Q (once per unit) and of the
//     K/V tiles into a ring of NSLOT shared-memory slots (full/empty
//     mbarriers, 128-byte swizzle);
//   * MMA warp: one thread issues tcgen05.mma S_s = Q_s K_j^T into tensor
//     memory and O_s += P_s V_j with P_s read from tensor memory; stage order
//     PV_0(j-1), S_0(j), PV_1(j-1), S_1(j) makes one tile's softmax overlap
//     the other tile's two GEMMs (the pages' ping-pong). That thread shares
//     its sub-partition with two softmax warps and waits for a scheduler slot
//     on every instruction, so its steady-state loop is kept short;
//   * softmax warpgroups (one per query tile, one thread per query row =
//     one TMEM lane): tcgen05.ld of the S row, mask, row max, conditional
//     rescale of O in tensor memory, exp2, row sum, P rounded to the input
//     type and written back over S with tcgen05.st; the same warps run the
//     epilogue (O / l, LSE) of their tile.
// The pages' intra-warpgroup overlap and named barriers have no direct
// counterpart: the MMA warp is asynchronous to the softmax warps by
// construction, and mbarriers + tcgen05.commit replace the named barriers.
//
// Tensor memory (512 columns x 128 lanes, FP32): S_s at column 128 s,
// O_s at 128 QST + D s.  16-bit P_s (64 columns) is written over the first
// columns of S_s after S_s has been read. FP8 with two query tiles writes P_s
// to one of two shared-memory buffers of its tile instead and releases S_s as
// soon as it is in registers, so the tile's next S GEMM runs while its softmax
// still computes P (order per key tile: S_0(j), PV_0(j-1), S_1(j), PV_1(j-1)).
//
// FP8 (E4M3) instance: per-128-token-block descales are applied to the
// logits per 128 x 128 tile; P is quantised to E4M3 with the V block's scale
// folded into the exponent (see softmax_tile); V arrives transposed
// ([B, Hkv, d, Nkpad], keys contiguous) so both GEMMs read K-major operands.
#pragma once

#include <cuda.h>
#include <math_constants.h>
#include <stdint.h>

#include <utility>

#include "ptx.cuh"

namespace attn {

enum : int { DT_F16 = 0, DT_BF16 = 1, DT_E4M3 = 2 };

// bit set in the device status word when a bounded wait expires
constexpr unsigned kStatusTimeout = 1u;
// cycles a wait may spin before the kernel gives up (about 2 s at 2 GHz)
constexpr long long kWaitBudgetCycles = 4000000000LL;

struct FwdParams {
  void* o;                 // [B, Nq, Hq, D], f16/bf16 (bf16 for the FP8 instance)
  float* lse;              // [B, Hq, Nq]
  const float* q_descale;  // FP8 only: [B, Hq, nqb]
  const float* k_descale;  //            [B, Hkv, nkb]
  const float* v_descale;  //            [B, Hkv, nkb]
  unsigned int* status;    // device status word
  int B, Hq, Hkv, group;   // group = Hq / Hkv
  int Nq, Nk;
  int n_kv_tiles;          // ceil(Nk / 128)
  int n_mblocks;           // ceil(Nq / (QST * 128))
  int n_units;             // B * Hq * n_mblocks
  int nqb, nkb;            // descale blocks per head
  float scale_log2;        // scale * log2(e)
  int active_stages;       // query tiles per unit that hold rows (1 when Nq <= 128)
  // split key ranges (non-causal only): unit = (head, row block, split); a
  // split covers split_tiles key tiles and writes FP32 partial results
  int n_splits;            // 1: no split, results go to o / lse
  int split_tiles;         // key tiles per split
  float* o_part;           // [n_splits, B, Hq, Nq, D] O / l of the split (n_splits > 1)
  // split instances: query heads packed into the rows of one tile (a GQA
  // group, or 1); tile row r is position m0 + r / pack_g of head hq + r % pack_g
  int pack_g;
  float* lse_part;         // [n_splits, B, Hq, Nq] natural-log LSE of the split
};

template <int D, int DT>
struct FwdCfg {
  static constexpr int ELT = (DT == DT_E4M3) ? 1 : 2;
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int QST = (D == 256) ? 1 : 2;   // query tiles per unit (TMEM budget)
  static constexpr int ROWB = D * ELT;              // bytes of one Q/K row
  // Q and K tiles: 128-byte swizzle in chunks of 128 bytes per row; a 64-byte
  // row (FP8, d = 64) is one chunk with the 64-byte swizzle
  static constexpr int SWZ = ROWB >= 128 ? 128 : 64;
  static constexpr int NCH = ROWB / SWZ;            // swizzle chunks per row
  static constexpr int CH_ELEMS = SWZ / ELT;        // elements per chunk
  static constexpr int CHUNK_BYTES = 128 * SWZ;     // one chunk of 128 rows
  static constexpr int QBYTES = BM * ROWB;
  static constexpr int KVBYTES = BN * ROWB;         // K tile; V (or V^T) tile is the same size
  static constexpr int SMEM_LIMIT = 232448;         // 227 KB opt-in per CTA
  static constexpr int SMEM_TAIL = 512;             // barriers + TMEM address + flags
  // FP8 with two query tiles: P goes to a shared-memory buffer per query tile
  // instead of over S in tensor memory, so the next S GEMM of a tile can run
  // while the softmax of its current key tile still computes P
  static constexpr bool PSMEM = (DT == DT_E4M3) && (QST == 2);
  static constexpr int PBYTES = BM * BN * ELT;      // one P tile (K-major, 128-byte swizzle)
  static constexpr int PTOTAL = PSMEM ? QST * 2 * PBYTES : 0;   // two buffers per query tile
  static constexpr int SLOT_FIT =
      (SMEM_LIMIT - 1024 - SMEM_TAIL - QST * QBYTES - PTOTAL) / KVBYTES;
  static constexpr int NSLOT = SLOT_FIT > 8 ? 8 : SLOT_FIT;
  static constexpr int SMEM_BYTES = 1024 + QST * QBYTES + PTOTAL + NSLOT * KVBYTES + SMEM_TAIL;
  static constexpr int TMEM_COLS = 512;
  static constexpr int S_COL0 = 0;                  // S_s at S_COL0 + 128 s
  static constexpr int O_COL0 = 128 * QST;          // O_s at O_COL0 + D s
  // two query tiles: 2 softmax warpgroups + one warpgroup holding the MMA and
  // TMA warps (and two idle warps) so registers can move between warpgroups
  static constexpr int NUM_WARPS = (QST == 2) ? 12 : 6;
  static constexpr int NTHREADS = NUM_WARPS * 32;
  static constexpr int W_MMA = QST * 4;
  static constexpr int W_LOAD = QST * 4 + 1;
  // register split (setmaxnreg) of the two-tile layout; the launch must give
  // each thread at least LAUNCH_REGS so that the split fits in the block's pool
  static constexpr int REG_SOFTMAX = 216;
  static constexpr int REG_OTHER = 72;
  static constexpr int LAUNCH_REGS = (2 * REG_SOFTMAX + REG_OTHER + 2) / 3;
  // softmax: lazy rescale threshold (log2 units) and exponent shift of P
  static constexpr float TAU = (DT == DT_E4M3) ? 2.0f : 8.0f;
  static constexpr float PSHIFT = (DT == DT_E4M3) ? 6.0f : 0.0f;

  static_assert(NSLOT >= 2, "shared memory too small for a double-buffered K/V ring");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory over budget");
  static_assert(O_COL0 + QST * D <= TMEM_COLS, "tensor memory over budget");
};

// ---------------------------------------------------------------- descriptors
// tcgen05 shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1 (bits 46-47).  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The same descriptor split into words: the high word (stride byte offset
// 1024, version, 128-byte swizzle) is the same for every operand here, and the
// start address is the low 14 bits of the low word in 16-byte units. Shared
// memory offsets stay below 2^18 bytes, so adding (offset >> 4) to the low
// word never carries out of the field: one add per MMA operand.
constexpr uint32_t kSdescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));
// the same for 64-byte rows: 64-byte swizzle (layout type 4), 8-row groups of 512 bytes
constexpr uint32_t kSdescHi64 = (512u >> 4) | (1u << (46 - 32)) | (4u << (61 - 32));
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}

// S = Q K^T: one MMA per 32 bytes of the head dimension; the operands' low
// descriptor words advance by the same offset in Q and K (16-byte units)
// (ACC0: the first MMA accumulates too; used for O += P V with P in shared
// memory; KPC: MMAs per swizzle chunk of a row; HI: descriptor high word)
template <int DT, int CHUNK_BYTES, bool ACC0 = false, int KPC = 4, uint32_t HI = kSdescHi,
          size_t... KK>
__device__ __forceinline__ void issue_s_mmas(uint32_t tS, uint32_t qlo, uint32_t klo, uint32_t idS,
                                             std::index_sequence<KK...>) {
  (ptx::mma_ss_lo<DT == DT_E4M3, ((KK > 0 || ACC0) ? 1 : 0),
                  (uint32_t)((((int)KK / KPC) * CHUNK_BYTES + ((int)KK % KPC) * 32) >> 4), HI>(
       tS, qlo, klo, idS),
   ...);
}
// O += P V with P read from tensor memory (8 columns per MMA) and the V tile
// advancing by VSTEP bytes per MMA; FIRST: the unit's first PV overwrites O
template <int DT, int VSTEP, bool FIRST, size_t... KK>
__device__ __forceinline__ void issue_pv_mmas(uint32_t tO, uint32_t tS, uint32_t vlo, uint32_t idO,
                                              std::index_sequence<KK...>) {
  (ptx::mma_ts_lo<DT == DT_E4M3, (FIRST && KK == 0) ? 0 : 1, (uint32_t)(KK * 8),
                  (uint32_t)((KK * VSTEP) >> 4), kSdescHi>(tO, tS, vlo, idO),
   ...);
}

// tcgen05 instruction descriptor: FP32 accumulate, dense, A K-major.
// fmt: 0 = f16 / e4m3, 1 = bf16 / e5m2 (per kind); b_mn_major selects a
// transposed (N-contiguous) B operand.
__host__ __device__ constexpr uint32_t idesc_make(uint32_t fmt, int M, int N, bool b_mn_major) {
  return (1u << 4)                          // D format: FP32
         | (fmt << 7)                       // A format
         | (fmt << 10)                      // B format
         | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ----------------------------------------------------------------- scheduling
struct Unit {
  int b, hq, hk, m0;   // hq: first query head of the unit; m0: first query position
  int j0;       // first key tile of the unit's key range
  int sp;       // split index
  int n_s[2];   // key tiles each query tile visits
  int n;        // max over the tiles
};

template <int QST, bool CAUSAL, bool SPLIT>
__device__ __forceinline__ Unit decode_unit(int u, const FwdParams& p) {
  Unit U;
  const int BH = p.B * p.Hq;
  int mb, bh;
  U.sp = 0;
  if (CAUSAL) {  // heaviest row blocks first, heads interleaved
    mb = p.n_mblocks - 1 - u / BH;
    bh = u % BH;
  } else {       // head-major (then row block, then split): concurrent CTAs share
                 // one head's K/V in L2, or stream disjoint ranges of it
    int v = u;
    if (SPLIT) {
      U.sp = u % p.n_splits;
      v = u / p.n_splits;
    }
    bh = v / p.n_mblocks;
    mb = v % p.n_mblocks;
  }
  const int G = SPLIT ? p.pack_g : 1;   // query heads per tile row group
  const int HP = p.Hq / G;                // packed head groups
  U.b = bh / HP;
  U.hq = (bh % HP) * G;
  U.hk = U.hq / p.group;
  U.m0 = mb * QST * (128 / G);
  U.j0 = SPLIT ? U.sp * p.split_tiles : 0;
  U.n = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    int n = p.n_kv_tiles - U.j0;
    if (SPLIT && p.split_tiles < n) n = p.split_tiles;
    if (CAUSAL) {
      const int last_row = U.m0 + s * 128 + 127;  // top-left aligned mask
      const int need = last_row / 128 + 1;
      n = need < n ? need : n;
    }
    const bool active = s < QST && (!SPLIT || s < p.active_stages);
    U.n_s[s] = active ? n : 0;
    if (active && n > U.n) U.n = n;
  }
  return U;
}

// unit visited by this CTA in round `it` (snake order for the causal case so
// that the CTA that took the heaviest unit of one round takes the lightest of
// the next); -1 when the round has no unit for this CTA, -2 when done
template <bool CAUSAL>
__device__ __forceinline__ int unit_of_round(int it, const FwdParams& p) {
  const int G = gridDim.x;
  const long long base = (long long)it * G;
  if (base >= p.n_units) return -2;
  const int c = (CAUSAL && (it & 1)) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const long long u = base + c;
  return u < p.n_units ? (int)u : -1;
}

// ------------------------------------------------------------ bounded waits
struct Ctl {
  volatile int* abort_flag;
  unsigned int* status;
};

// suspend-time hint of a waiting thread: waiters sleep in hardware instead of
// spinning, so they do not take issue slots from the warps doing the work
constexpr uint32_t kWaitSuspendNs = 200000;

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kWaitSuspendNs)) return true;
    if (*ctl.abort_flag) return false;
    if (clock64() - t0 > kWaitBudgetCycles) {
      *ctl.abort_flag = 1;
      atomicOr(ctl.status, kStatusTimeout);
      return false;
    }
  }
}

// a whole warp waits; the outcome is made warp-uniform so that the
// warp-collective tcgen05 loads/stores that follow stay convergent
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  const bool ok = wait_bar(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// The softmax warps' wait for S: polled without the suspend hint and without
// reading the abort flag inside the loop (measured: waking a suspended warp,
// or the extra poll, costs 2-4 % of the forward's time on this wait, which
// sits on the softmax's critical path). Still bounded by the cycle budget; on
// expiry it flags the timeout like wait_bar. After another role aborted, it
// gives up when its own budget runs out.
__device__ __forceinline__ bool warp_spin_wait_bar(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  bool ok = true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitBudgetCycles) {
      ok = false;
      break;
    }
  }
  if (!ok) {
    *ctl.abort_flag = 1;
    atomicOr(ctl.status, kStatusTimeout);
  }
  return __all_sync(0xffffffffu, ok);
}

// 8 x 8 transpose of 16-byte pieces (w[4k .. 4k+3] = piece k) inside each
// octet of lanes: afterwards piece k of lane 8g + i is what piece i of lane
// 8g + k was. Three butterfly stages, each swapping the off-diagonal 4 x 4,
// 2 x 2 and 1 x 1 blocks of pieces between lanes that differ in one bit.
__device__ __forceinline__ void octet_transpose(uint32_t (&w)[32], int lane) {
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k & m) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t send = hi ? w[4 * k + e] : w[4 * (k | m) + e];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        if (hi)
          w[4 * k + e] = recv;
        else
          w[4 * (k | m) + e] = recv;
      }
    }
  }
}

// --------------------------------------------------------------------- kernel
template <int D, int DT, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<D, DT>::NTHREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D, DT>;
  constexpr int QST = C::QST;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = ptx::smem_addr(smem_raw);
  const uint32_t pad = (1024u - (sraw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  static_assert(!(C::PSMEM && SPLIT), "split instances keep P in tensor memory");
  const uint32_t sQ = sraw + pad;                       // QST query tiles
  const uint32_t sP = sQ + QST * C::QBYTES;             // P tiles (shared-memory P only)
  const uint32_t sKV = sP + C::PTOTAL;                  // NSLOT K/V slots
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + QST * C::QBYTES + C::PTOTAL + NSLOT * C::KVBYTES);

  // barrier table
  constexpr int B_QFULL = 0;                 // [2]   TMA Q landed            (tx)
  constexpr int B_QEMPTY = 2;                // [1]   last S GEMM of unit done (commit)
  constexpr int B_KVFULL = 3;                // [NSLOT] TMA K/V landed        (tx)
  constexpr int B_KVEMPTY = 3 + NSLOT;       // [NSLOT] GEMMs reading slot done (commit)
  constexpr int B_SFULL = 3 + 2 * NSLOT;     // [2]   S_s ready               (commit)
  constexpr int B_PFULL = B_SFULL + 2;       // [2]   P_s written, O_s rescaled (4 warp arrivals)
  constexpr int B_OFULL = B_PFULL + 2;       // [2]   last PV of unit done    (commit)
  constexpr int B_OEMPTY = B_OFULL + 2;      // [2]   epilogue read O_s       (4 warp arrivals)
  constexpr int B_DRAIN = B_OEMPTY + 2;      // [1]   all MMAs of this CTA done (commit)
  // shared-memory P only: P buffer b of tile s is entry 2 s + b
  constexpr int B_SFREE = B_DRAIN + 1;       // [2]   S_s read into registers (4 warp arrivals)
  constexpr int B_PFULLB = B_SFREE + 2;      // [2x2] P buffer written      (4 warp arrivals)
  constexpr int B_PFREEB = B_PFULLB + 4;     // [2x2] PV done reading it    (commit)
  constexpr int NBARS = B_PFREEB + 4;
  static_assert(NBARS * 8 + 16 <= C::SMEM_TAIL, "barrier table too large");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) -> uint32_t { return ptx::smem_addr(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Ctl ctl{abort_flag, p.status};
  // query tiles that hold rows: only the split (decode) instances skip an
  // all-padding second tile; the others keep the count a compile-time constant
  const int n_active = SPLIT ? (QST < p.active_stages ? QST : p.active_stages) : QST;
  const int G = SPLIT ? p.pack_g : 1;   // query heads packed per tile row group

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(B_QFULL + s), 1);
      ptx::mbar_init(bar(B_SFULL + s), 1);
      ptx::mbar_init(bar(B_PFULL + s), 4);   // one elected arrival per softmax warp
      ptx::mbar_init(bar(B_OFULL + s), 1);
      ptx::mbar_init(bar(B_OEMPTY + s), 4);
    }
    ptx::mbar_init(bar(B_QEMPTY), 1);
    for (int i = 0; i < NSLOT; ++i) {
      ptx::mbar_init(bar(B_KVFULL + i), 1);
      ptx::mbar_init(bar(B_KVEMPTY + i), 1);
    }
    ptx::mbar_init(bar(B_DRAIN), 1);
    for (int s = 0; s < 2; ++s) ptx::mbar_init(bar(B_SFREE + s), 4);
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(bar(B_PFULLB + i), 4);
      ptx::mbar_init(bar(B_PFREEB + i), 1);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == C::W_MMA) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == C::W_LOAD && lane == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_LOAD) {
    // ===================================================== TMA producer
    if constexpr (QST == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if (lane == 0) {
      int kv_it = 0, u_it = 0;
      bool ok = true;
      const uint64_t pol_kv = ptx::policy_evict_last();
      for (int it = 0; ok; ++it) {
        const int u = unit_of_round<CAUSAL>(it, p);
        if (u == -2) break;
        if (u < 0) continue;
        const Unit U = decode_unit<QST, CAUSAL, SPLIT>(u, p);
        ok = wait_bar(bar(B_QEMPTY), (u_it & 1) ^ 1, ctl);
        if (!ok) break;
        for (int s = 0; s < n_active; ++s) {
          ptx::mbar_arrive_expect_tx(bar(B_QFULL + s), C::QBYTES);
          for (int ch = 0; ch < C::NCH; ++ch)
            ptx::tma_load_4d(sQ + s * C::QBYTES + ch * C::CHUNK_BYTES, &tmQ, bar(B_QFULL + s),
                             ch * C::CH_ELEMS, U.hq, U.m0 + s * (128 / G), U.b);
        }
        for (int j = 0; j < U.n && ok; ++j) {
          // K_j
          {
            const int slot = kv_it % NSLOT;
            ok = wait_bar(bar(B_KVEMPTY + slot), ((kv_it / NSLOT) & 1) ^ 1, ctl);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(B_KVFULL + slot), C::KVBYTES);
            for (int ch = 0; ch < C::NCH; ++ch)
              ptx::tma_load_4d_hint(sKV + slot * C::KVBYTES + ch * C::CHUNK_BYTES, &tmK,
                                    bar(B_KVFULL + slot), ch * C::CH_ELEMS, U.hk,
                                    (U.j0 + j) * 128, U.b, pol_kv);
            ++kv_it;
          }
          // V_j (FP8: one box of the transposed tensor, D rows x 128 keys)
          {
            const int slot = kv_it % NSLOT;
            ok = wait_bar(bar(B_KVEMPTY + slot), ((kv_it / NSLOT) & 1) ^ 1, ctl);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(B_KVFULL + slot), C::KVBYTES);
            if constexpr (DT == DT_E4M3) {
              ptx::tma_load_4d_hint(sKV + slot * C::KVBYTES, &tmV, bar(B_KVFULL + slot),
                                    (U.j0 + j) * 128, 0, U.hk, U.b, pol_kv);
            } else {
              for (int ch = 0; ch < C::NCH; ++ch)
                ptx::tma_load_4d_hint(sKV + slot * C::KVBYTES + ch * C::CHUNK_BYTES, &tmV,
                                      bar(B_KVFULL + slot), ch * C::CH_ELEMS, U.hk,
                                      (U.j0 + j) * 128, U.b, pol_kv);
            }
            ++kv_it;
          }
        }
        ++u_it;
      }
      // wait (bounded) for copies still in flight before the CTA can exit
      const int pending = kv_it < NSLOT ? kv_it : NSLOT;
      for (int t = kv_it - pending; t < kv_it; ++t)
        wait_bar(bar(B_KVFULL + t % NSLOT), (t / NSLOT) & 1, Ctl{abort_flag, p.status});
      if (u_it > 0)
        for (int s = 0; s < n_active; ++s)
          wait_bar(bar(B_QFULL + s), (u_it - 1) & 1, ctl);
    }
    __syncwarp();
  } else if (warp == C::W_MMA) {
    // ===================================================== MMA issuer
    if constexpr (QST == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if (lane == 0) {
      constexpr uint32_t fmt = (DT == DT_BF16) ? 1u : 0u;
      constexpr uint32_t idS = idesc_make(fmt, 128, 128, false);
      constexpr uint32_t idO = idesc_make(fmt, 128, D, DT != DT_E4M3);
      // S = Q K^T into tS and O += P V with P read from tS (accumulating),
      // from the low descriptor words of the operands' shared-memory tiles
      auto issue_s = [&](uint32_t tS, uint32_t qlo, uint32_t klo) {
        issue_s_mmas<DT, C::CHUNK_BYTES, false, C::SWZ / 32, C::SWZ == 128 ? kSdescHi : kSdescHi64>(
            tS, qlo, klo, idS, std::make_index_sequence<C::ROWB / 32>{});
      };
      // FP8: 32 keys per MMA (V^T tile, K-major); 16-bit: 16 keys per MMA
      constexpr int PV_MMAS = DT == DT_E4M3 ? 4 : 8;
      constexpr int VSTEP = DT == DT_E4M3 ? 32 : 2048;
      auto issue_pv = [&](uint32_t tO, uint32_t tS, uint32_t vlo) {
        issue_pv_mmas<DT, VSTEP, false>(tO, tS, vlo, idO, std::make_index_sequence<PV_MMAS>{});
      };
      auto issue_pv_first = [&](uint32_t tO, uint32_t tS, uint32_t vlo) {
        issue_pv_mmas<DT, VSTEP, true>(tO, tS, vlo, idO, std::make_index_sequence<PV_MMAS>{});
      };
      if constexpr (C::PSMEM) {
        // P in shared memory (two buffers per query tile): per key tile j the
        // order is S_0(j), PV_0(j-1), S_1(j), PV_1(j-1). S_s(j) waits only
        // until the softmax of tile s holds S_s(j-1) in registers, so it runs
        // while that softmax still computes P_s(j-1); PV reads P from shared
        // memory and its completion frees the buffer. PV number n of a tile
        // uses buffer n % 2, whose barriers complete once per two PVs.
        int kv_it = 0, u_it = 0;
        int pv_cnt[2] = {0, 0};   // PV GEMMs issued per query tile
        int sg_cnt[2] = {0, 0};   // S GEMMs issued per query tile
        bool ok = true;
        const uint32_t qlo0 = sdesc_lo(sQ, 16);
        const uint32_t plo0 = sdesc_lo(sP, 16);   // buffer i at plo0 + i * (PBYTES >> 4)
        auto pv_ss = [&](int s, int n, bool first, uint32_t vlo) {
          const uint32_t tO = tmem + C::O_COL0 + D * s;
          const uint32_t plo = plo0 + (uint32_t)(2 * s + (n & 1)) * (C::PBYTES >> 4);
          if (first)
            issue_s_mmas<DT, C::CHUNK_BYTES, false>(tO, plo, vlo, idO,
                                                    std::make_index_sequence<C::BN * C::ELT / 32>{});
          else
            issue_s_mmas<DT, C::CHUNK_BYTES, true>(tO, plo, vlo, idO,
                                                   std::make_index_sequence<C::BN * C::ELT / 32>{});
          ptx::tc_commit(bar(B_PFREEB + 2 * s + (n & 1)));
        };
        for (int it = 0; ok; ++it) {
          const int u = unit_of_round<CAUSAL>(it, p);
          if (u == -2) break;
          if (u < 0) continue;
          const Unit U = decode_unit<QST, CAUSAL, SPLIT>(u, p);
          for (int s = 0; s < QST && ok; ++s) ok = wait_bar(bar(B_QFULL + s), u_it & 1, ctl);
          if (!ok) break;
          ptx::tc_fence_after();
          const int n_both = U.n_s[0] < U.n_s[1] ? U.n_s[0] : U.n_s[1];
          const int jend = n_both - 1;
          for (int j = 0; j <= U.n && ok; ++j) {
            if (j == 2 && jend > 2) {
              // steady state: both tiles take S(j) and PV(j-1), no unit edge
              // step in range; running counters, one status check per tile
              int vs = (kv_it + 3) % NSLOT;
              uint32_t vph = ((kv_it + 3) / NSLOT) & 1;
              int ks = (kv_it + 4) % NSLOT;
              uint32_t kph = ((kv_it + 4) / NSLOT) & 1;
              uint32_t sf0 = (sg_cnt[0] - 1) & 1, sf1 = (sg_cnt[1] - 1) & 1;
              int n0 = pv_cnt[0], n1 = pv_cnt[1];
              const uint32_t tS0 = tmem + C::S_COL0, tS1 = tS0 + 128;
              bool sok = true;
              for (; j < jend; ++j) {
                const uint32_t klo = sdesc_lo(sKV + ks * C::KVBYTES, 16);
                const uint32_t vlo = sdesc_lo(sKV + vs * C::KVBYTES, 16);
                sok &= wait_bar(bar(B_KVFULL + ks), kph, ctl);
                sok &= wait_bar(bar(B_SFREE + 0), sf0, ctl);
                ptx::tc_fence_after();
                issue_s(tS0, qlo0, klo);
                ptx::tc_commit(bar(B_SFULL + 0));
                sok &= wait_bar(bar(B_KVFULL + vs), vph, ctl);
                sok &= wait_bar(bar(B_PFULLB + (n0 & 1)), (n0 >> 1) & 1, ctl);
                ptx::tc_fence_after();
                pv_ss(0, n0, false, vlo);
                sok &= wait_bar(bar(B_SFREE + 1), sf1, ctl);
                ptx::tc_fence_after();
                issue_s(tS1, qlo0 + (C::QBYTES >> 4), klo);
                ptx::tc_commit(bar(B_SFULL + 1));
                ptx::tc_commit(bar(B_KVEMPTY + ks));
                sok &= wait_bar(bar(B_PFULLB + 2 + (n1 & 1)), (n1 >> 1) & 1, ctl);
                ptx::tc_fence_after();
                pv_ss(1, n1, false, vlo);
                ptx::tc_commit(bar(B_KVEMPTY + vs));
                sf0 ^= 1u;
                sf1 ^= 1u;
                ++n0;
                ++n1;
                vs = ks + 1;
                vph = kph;
                if (vs == NSLOT) {
                  vs = 0;
                  vph ^= 1u;
                }
                ks = vs + 1;
                kph = vph;
                if (ks == NSLOT) {
                  ks = 0;
                  kph ^= 1u;
                }
                if (!sok) break;
              }
              sg_cnt[0] += n0 - pv_cnt[0];
              sg_cnt[1] += n1 - pv_cnt[1];
              pv_cnt[0] = n0;
              pv_cnt[1] = n1;
              ok = sok;
              if (!ok) break;
            }
            const int k_idx = kv_it + 2 * j;       // ring index of K_j
            const int v_idx = kv_it + 2 * j - 1;   // ring index of V_{j-1}
            const int kslot = k_idx % NSLOT;
            const int vslot = (v_idx + NSLOT) % NSLOT;
            bool k_ready = false, v_ready = false;
#pragma unroll
            for (int s = 0; s < QST; ++s) {
              if (j < U.n_s[s]) {
                // S_s = Q_s K_j^T once the softmax holds S_s(j-1)
                if (!k_ready) {
                  ok = wait_bar(bar(B_KVFULL + kslot), (k_idx / NSLOT) & 1, ctl);
                  k_ready = true;
                }
                if (ok && sg_cnt[s] > 0) ok = wait_bar(bar(B_SFREE + s), (sg_cnt[s] - 1) & 1, ctl);
                if (!ok) break;
                ptx::tc_fence_after();
                issue_s(tmem + C::S_COL0 + 128 * s, qlo0 + (uint32_t)s * (C::QBYTES >> 4),
                        sdesc_lo(sKV + kslot * C::KVBYTES, 16));
                ptx::tc_commit(bar(B_SFULL + s));
                ++sg_cnt[s];
                // the second query tile visits every key tile: it is the last reader
                if (s == QST - 1) ptx::tc_commit(bar(B_KVEMPTY + kslot));
              }
              if (j >= 1 && j - 1 < U.n_s[s]) {
                // O_s += P_s V_{j-1}, P_s from shared memory
                if (!v_ready) {
                  ok = wait_bar(bar(B_KVFULL + vslot), (v_idx / NSLOT) & 1, ctl);
                  v_ready = true;
                }
                const int n = pv_cnt[s];
                if (ok) ok = wait_bar(bar(B_PFULLB + 2 * s + (n & 1)), (n >> 1) & 1, ctl);
                if (ok && j == 1) ok = wait_bar(bar(B_OEMPTY + s), (u_it & 1) ^ 1, ctl);
                if (!ok) break;
                ptx::tc_fence_after();
                pv_ss(s, n, j == 1, sdesc_lo(sKV + vslot * C::KVBYTES, 16));
                ++pv_cnt[s];
                if (j - 1 == U.n_s[s] - 1) ptx::tc_commit(bar(B_OFULL + s));
                if (s == QST - 1) ptx::tc_commit(bar(B_KVEMPTY + vslot));
              }
            }
            if (!ok) break;
            if (j == U.n - 1) ptx::tc_commit(bar(B_QEMPTY));
          }
          kv_it += 2 * U.n;
          ++u_it;
        }
      } else {
      int kv_it = 0, u_it = 0;
      int pv_cnt[2] = {0, 0};
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int u = unit_of_round<CAUSAL>(it, p);
        if (u == -2) break;
        if (u < 0) continue;
        const Unit U = decode_unit<QST, CAUSAL, SPLIT>(u, p);
        for (int s = 0; s < n_active && ok; ++s)
          ok = wait_bar(bar(B_QFULL + s), u_it & 1, ctl);
        const int s_last = n_active - 1;
        if (!ok) break;
        ptx::tc_fence_after();
        for (int j = 0; j <= U.n && ok; ++j) {
          if constexpr (QST == 2 && !SPLIT) {
            // Steady state: for 2 <= j < min(n_s) - 1 both query tiles take
            // PV(j-1) and S(j) and none of the unit's first or last steps
            // (O buffers, Q release, last PV) falls in the range. The issuing
            // thread shares its sub-partition with two softmax warps and
            // waits for a scheduler slot on every instruction, so this loop
            // keeps ring slots and phases as running counters, tests no edge
            // case and checks the waits' status once per key tile.
            const int n_both = U.n_s[0] < U.n_s[1] ? U.n_s[0] : U.n_s[1];
            const int jend = n_both - 1;
            if (j == 2 && jend > 2) {
              int vs = (kv_it + 3) % NSLOT;                 // V_{j-1}: ring index kv_it + 2j - 1
              uint32_t vph = ((kv_it + 3) / NSLOT) & 1;
              int ks = (kv_it + 4) % NSLOT;                 // K_j: ring index kv_it + 2j
              uint32_t kph = ((kv_it + 4) / NSLOT) & 1;
              uint32_t pph0 = pv_cnt[0] & 1, pph1 = pv_cnt[1] & 1;
              const uint32_t qlo0 = sdesc_lo(sQ, 16);
              const uint32_t qlo1 = sdesc_lo(sQ + C::QBYTES, 16);
              const uint32_t tS0 = tmem + C::S_COL0, tS1 = tS0 + 128;
              const uint32_t tO0 = tmem + C::O_COL0, tO1 = tO0 + D;
              bool sok = true;
              for (; j < jend; ++j) {
                const uint32_t vlo = sdesc_lo(sKV + vs * C::KVBYTES, DT == DT_E4M3 ? 16 : C::CHUNK_BYTES);
                const uint32_t klo = sdesc_lo(sKV + ks * C::KVBYTES, 16);
                sok &= wait_bar(bar(B_KVFULL + vs), vph, ctl);
                sok &= wait_bar(bar(B_PFULL + 0), pph0, ctl);
                ptx::tc_fence_after();
                issue_pv(tO0, tS0, vlo);
                sok &= wait_bar(bar(B_KVFULL + ks), kph, ctl);
                ptx::tc_fence_after();
                issue_s(tS0, qlo0, klo);
                ptx::tc_commit(bar(B_SFULL + 0));
                sok &= wait_bar(bar(B_PFULL + 1), pph1, ctl);
                ptx::tc_fence_after();
                issue_pv(tO1, tS1, vlo);
                ptx::tc_commit(bar(B_KVEMPTY + vs));
                issue_s(tS1, qlo1, klo);
                ptx::tc_commit(bar(B_SFULL + 1));
                ptx::tc_commit(bar(B_KVEMPTY + ks));
                pph0 ^= 1u;
                pph1 ^= 1u;
                vs = ks + 1;
                vph = kph;
                if (vs == NSLOT) {
                  vs = 0;
                  vph ^= 1u;
                }
                ks = vs + 1;
                kph = vph;
                if (ks == NSLOT) {
                  ks = 0;
                  kph ^= 1u;
                }
                if (!sok) break;
              }
              pv_cnt[0] += j - 2;
              pv_cnt[1] += j - 2;
              ok = sok;
              if (!ok) break;
            }
          }
          if constexpr (QST == 1 && !SPLIT) {
            // the same steady state with one query tile: PV(j-1), S(j)
            const int jend = U.n_s[0] - 1;
            if (j == 2 && jend > 2) {
              int vs = (kv_it + 3) % NSLOT;
              uint32_t vph = ((kv_it + 3) / NSLOT) & 1;
              int ks = (kv_it + 4) % NSLOT;
              uint32_t kph = ((kv_it + 4) / NSLOT) & 1;
              uint32_t pph = pv_cnt[0] & 1;
              const uint32_t qlo0 = sdesc_lo(sQ, 16);
              const uint32_t tS0 = tmem + C::S_COL0, tO0 = tmem + C::O_COL0;
              bool sok = true;
              for (; j < jend; ++j) {
                const uint32_t vlo = sdesc_lo(sKV + vs * C::KVBYTES, DT == DT_E4M3 ? 16 : C::CHUNK_BYTES);
                const uint32_t klo = sdesc_lo(sKV + ks * C::KVBYTES, 16);
                sok &= wait_bar(bar(B_KVFULL + vs), vph, ctl);
                sok &= wait_bar(bar(B_PFULL + 0), pph, ctl);
                ptx::tc_fence_after();
                issue_pv(tO0, tS0, vlo);
                ptx::tc_commit(bar(B_KVEMPTY + vs));
                sok &= wait_bar(bar(B_KVFULL + ks), kph, ctl);
                ptx::tc_fence_after();
                issue_s(tS0, qlo0, klo);
                ptx::tc_commit(bar(B_SFULL + 0));
                ptx::tc_commit(bar(B_KVEMPTY + ks));
                pph ^= 1u;
                vs = ks + 1;
                vph = kph;
                if (vs == NSLOT) {
                  vs = 0;
                  vph ^= 1u;
                }
                ks = vs + 1;
                kph = vph;
                if (ks == NSLOT) {
                  ks = 0;
                  kph ^= 1u;
                }
                if (!sok) break;
              }
              pv_cnt[0] += j - 2;
              ok = sok;
              if (!ok) break;
            }
          }
          const int k_idx = kv_it + 2 * j;       // ring index of K_j
          const int v_idx = kv_it + 2 * j - 1;   // ring index of V_{j-1}
          const int kslot = k_idx % NSLOT;
          const int vslot = (v_idx + NSLOT) % NSLOT;
          bool k_ready = false, v_ready = false;
#pragma unroll
          for (int s = 0; s < QST; ++s) {
            const uint32_t tS = tmem + C::S_COL0 + 128 * s;
            const uint32_t tO = tmem + C::O_COL0 + D * s;
            if (j >= 1 && j - 1 < U.n_s[s]) {
              // O_s += P_s V_{j-1}
              if (!v_ready) {
                ok = wait_bar(bar(B_KVFULL + vslot), (v_idx / NSLOT) & 1, ctl);
                v_ready = true;
              }
              if (ok) ok = wait_bar(bar(B_PFULL + s), pv_cnt[s] & 1, ctl);
              ++pv_cnt[s];
              if (ok && j == 1) ok = wait_bar(bar(B_OEMPTY + s), (u_it & 1) ^ 1, ctl);
              if (!ok) break;
              ptx::tc_fence_after();
              const uint32_t vbase = sKV + vslot * C::KVBYTES;
              if constexpr (SPLIT) {
                // (the split instances' issuing thread has no registers to spare
                // for the precomputed descriptor words)
#pragma unroll
                for (int kk = 0; kk < (DT == DT_E4M3 ? 4 : 8); ++kk) {
                  if constexpr (DT == DT_E4M3)
                    ptx::mma_f8_ts(tO, tS + kk * 8, sdesc_sw128(vbase + kk * 32, 16, 1024), idO,
                                   (j > 1 || kk > 0) ? 1u : 0u);
                  else
                    ptx::mma_f16_ts(tO, tS + kk * 8,
                                    sdesc_sw128(vbase + kk * 2048, C::CHUNK_BYTES, 1024), idO,
                                    (j > 1 || kk > 0) ? 1u : 0u);
                }
              } else {
                const uint32_t vlo = sdesc_lo(vbase, DT == DT_E4M3 ? 16 : C::CHUNK_BYTES);
                if (j > 1) issue_pv(tO, tS, vlo);
                else issue_pv_first(tO, tS, vlo);
              }
              if (j - 1 == U.n_s[s] - 1) ptx::tc_commit(bar(B_OFULL + s));
              // the last active query tile visits every key tile: it is the last reader
              if (s == s_last) ptx::tc_commit(bar(B_KVEMPTY + vslot));
            }
            if (j < U.n_s[s]) {
              // S_s = Q_s K_j^T
              if (!k_ready) {
                ok = wait_bar(bar(B_KVFULL + kslot), (k_idx / NSLOT) & 1, ctl);
                k_ready = true;
                if (!ok) break;
                ptx::tc_fence_after();
              }
              const uint32_t qbase = sQ + s * C::QBYTES;
              const uint32_t kbase = sKV + kslot * C::KVBYTES;
              constexpr int KSTEPS = C::ROWB / 32;   // 32 bytes of K per MMA
              if constexpr (SPLIT) {
                // (the split instances' issuing thread has no registers to spare
                // for the precomputed descriptor words)
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                  const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
                  const uint64_t a = sdesc_sw128(qbase + off, 16, 1024);
                  const uint64_t b = sdesc_sw128(kbase + off, 16, 1024);
                  if constexpr (DT == DT_E4M3)
                    ptx::mma_f8_ss(tS, a, b, idS, kk > 0 ? 1u : 0u);
                  else
                    ptx::mma_f16_ss(tS, a, b, idS, kk > 0 ? 1u : 0u);
                }
              } else {
                issue_s(tS, sdesc_lo(qbase, 16), sdesc_lo(kbase, 16));
              }
              ptx::tc_commit(bar(B_SFULL + s));
              if (s == s_last) ptx::tc_commit(bar(B_KVEMPTY + kslot));
            }
          }
          if (!ok) break;
          if (j == U.n - 1) ptx::tc_commit(bar(B_QEMPTY));
        }
        kv_it += 2 * U.n;
        ++u_it;
      }
      }
      // every MMA issued by this thread must finish before TMEM is released
      ptx::tc_commit(bar(B_DRAIN));
      wait_bar(bar(B_DRAIN), 0, Ctl{abort_flag, p.status});
    }
    __syncwarp();
  } else if (warp < QST * 4) {
    // ===================================================== softmax warpgroups
    if constexpr (QST == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    const int s = warp >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane; // row within the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL0 + 128 * s;
    const uint32_t tO = tmem + lane_off + C::O_COL0 + D * s;
    int s_cnt = 0, u_it = 0;
    int p_cnt = 0;   // P tiles this warpgroup has handed to the MMA thread
    // shared-memory P: this thread's row of the tile's P buffer (K-major,
    // 128-byte swizzle: 8-row groups of 1024 bytes, 128 bytes per row)
    const uint32_t prow0 = sP + 2 * s * C::PBYTES + (r >> 3) * 1024 + (r & 7) * 128;
    bool ok = true;
    // a query tile that holds no rows in this launch (Nq <= 128) does nothing
    for (int it = 0; ok && s < n_active; ++it) {
      const int u = unit_of_round<CAUSAL>(it, p);
      if (u == -2) break;
      if (u < 0) continue;
      const Unit U = decode_unit<QST, CAUSAL, SPLIT>(u, p);
      const int m_s = U.m0 + s * (128 / G);   // first query position of this tile
      const int row = m_s + r / G;            // query position of this thread's row
      const int hrow = U.hq + r % G;          // query head of this thread's row
      const int ns = s == 0 ? U.n_s[0] : U.n_s[1];   // (no dynamic index: U stays in registers)

      float qd = 1.f, vref = 1.f;
      const float* kd_row = nullptr;
      const float* vd_row = nullptr;
      if constexpr (DT == DT_E4M3) {
        const int qb = m_s >> 7;
        qd = (qb < p.nqb) ? __ldg(p.q_descale + ((long long)U.b * p.Hq + U.hq) * p.nqb + qb) : 1.f;
        kd_row = p.k_descale + ((long long)U.b * p.Hkv + U.hk) * p.nkb;
        vd_row = p.v_descale + ((long long)U.b * p.Hkv + U.hk) * p.nkb;
        float vm = 0.f;
        for (int t = lane; t < p.nkb; t += 32) vm = fmaxf(vm, __ldg(vd_row + t));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
        vref = vm > 0.f ? vm : 1.f;
      }

      float mi = -CUDART_INF_F;   // running max of the scaled logits (log2 units)
      float li = 0.f;             // running sum of exp2(logit - mi)
      // FP8: descales of the next key tile are loaded one iteration ahead so
      // their latency stays off the softmax critical path
      // FP8: the per-tile factors of tile j (logit scale, exponent bias, sum
      // scale) are computed at the end of tile j-1, from descales loaded a
      // tile earlier still, so neither the loads nor the divisions sit on
      // the softmax critical path
      float cj_cur = p.scale_log2, bias_cur = 0.f, ssc_cur = 1.f;
      float kd_next = 1.f, vd_next = 1.f;
      // (no divisions: with the softmax warps on every sub-partition busy,
      // each of the few scalar instructions between two tiles costs cycles
      // that no other work hides)
      const float cq = p.scale_log2 * qd;
      const float lvref = ptx::lg2(vref);
      auto fp8_factors = [&](float kd, float vd, float& cjo, float& bo, float& sso) {
        const float lr = ptx::lg2(vd) - lvref;   // log2 of V block scale / largest, <= 0
        cjo = cq * kd;
        bo = C::PSHIFT + lr;
        sso = ptx::ex2(-lr);
      };
      if constexpr (DT == DT_E4M3) {
        fp8_factors(__ldg(kd_row + U.j0), __ldg(vd_row + U.j0), cj_cur, bias_cur, ssc_cur);
        if (ns > 1) {
          kd_next = __ldg(kd_row + U.j0 + 1);
          vd_next = __ldg(vd_row + U.j0 + 1);
        }
      }
      for (int j = 0; j < ns; ++j) {
        ok = warp_spin_wait_bar(bar(B_SFULL + s), s_cnt & 1, ctl);
        ++s_cnt;
        if (!ok) break;
        ptx::tc_fence_after();
        // full tiles: the row maximum comes with the TMEM load (tcgen05.ld.red);
        // a tile with masked keys (causal diagonal, ragged key tail) takes the
        // maximum of its unmasked logits after the mask instead. Long runs of
        // max instructions on the softmax warps also take the issue slots the
        // MMA-issuing thread needs.
        const int n0 = (U.j0 + j) * 128;
        const bool masked = (n0 + 128 > p.Nk) || (CAUSAL && n0 + 127 > m_s);
        uint32_t sr[128];
        float rmax;
        if (!masked) ptx::tmem_ld_max_x128(tS, sr, rmax);
        else ptx::tmem_ld_x128(tS, sr);
        if constexpr (C::PSMEM) {
          // S_s is in registers: the next S GEMM of this tile may overwrite it
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(B_SFREE + s));
        }
        float sv[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(sr[c]);

        if (masked) {
          int lim = p.Nk - n0;
          if (CAUSAL) lim = min(lim, row - n0 + 1);
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c < lim) ? sv[c] : -CUDART_INF_F;
          // 16 independent chains of 3-input max, then a tree
          float mx[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            mx[i] = ptx::max3(sv[i], sv[i + 16], sv[i + 32]);
            mx[i] = ptx::max3(mx[i], sv[i + 48], sv[i + 64]);
            mx[i] = ptx::max3(mx[i], sv[i + 80], sv[i + 96]);
            mx[i] = fmaxf(mx[i], sv[i + 112]);
          }
          const float mxa = ptx::max3(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], mx[5]),
                                      ptx::max3(mx[6], mx[7], mx[8]));
          const float mxb = ptx::max3(ptx::max3(mx[9], mx[10], mx[11]),
                                      ptx::max3(mx[12], mx[13], mx[14]), mx[15]);
          rmax = fmaxf(mxa, mxb);
        }

        const float cj = cj_cur;           // logit scale of this tile (log2 units)
        const float bias_extra = bias_cur; // FP8: exponent shift and V-block factor
        const float sum_scale = ssc_cur;   // FP8: converts the tile's row sum back to unit P
        const float mj = rmax * cj;
        const float m_new = fmaxf(mi, mj);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          mi = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        } else if (m_new > mi + C::TAU) {
          // the new maximum exceeds the reference by more than 2^TAU:
          // move the reference (merge rule of section 4.2) and rescale O, l
          alpha = ptx::ex2(mi - m_new);
          mi = m_new;
          li *= alpha;
          rescale = true;
        }
        const bool any_rescale = __any_sync(0xffffffffu, rescale);
        if constexpr (C::PSMEM) {
          // P buffer p_cnt % 2 is free once PV number p_cnt - 2 is done; a
          // rescale of O waits until after P is written (below)
          if (p_cnt >= 2) {
            const int n = p_cnt - 2;
            ok = warp_wait_bar(bar(B_PFREEB + 2 * s + (n & 1)), (n >> 1) & 1, ctl);
            if (!ok) break;
            ptx::tc_fence_after();
          }
        } else if (any_rescale) {
#pragma unroll 1
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t o32[32];
            ptx::tmem_ld_x32(tO + cb, o32);
#pragma unroll
            for (int c = 0; c < 32; ++c) o32[c] = __float_as_uint(__uint_as_float(o32[c]) * alpha);
            ptx::tmem_st_x32(tO + cb, o32);
          }
        }

        // P = exp2(logit - reference), row sum, write P over S in 32-column
        // chunks as they are produced (the whole S row is already in registers)
        const float nbias = bias_extra - mi;
        float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
        const uint32_t prow = prow0 + (uint32_t)(p_cnt & 1) * C::PBYTES;   // shared-memory P
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int c = 32 * k; c < 32 * k + 32; c += 4) {
            float x0, x1, x2, x3;
            ptx::fma2(x0, x1, sv[c], sv[c + 1], cj, cj, nbias, nbias);
            ptx::fma2(x2, x3, sv[c + 2], sv[c + 3], cj, cj, nbias, nbias);
            sv[c] = ptx::ex2(x0);
            sv[c + 1] = ptx::ex2(x1);
            sv[c + 2] = ptx::ex2(x2);
            sv[c + 3] = ptx::ex2(x3);
            ptx::add2(sum0, sum1, sv[c], sv[c + 1]);
            ptx::add2(sum2, sum3, sv[c + 2], sv[c + 3]);
          }
          if constexpr (DT == DT_E4M3) {
            uint32_t pk[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int e = 32 * k + 4 * c;
              pk[c] = ptx::pack_e4m3x4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
            }
            if constexpr (C::PSMEM) {
              // keys 32k .. 32k+31 are the 16-byte chunks 2k, 2k+1 of the row
              // (K-major, 128-byte swizzle: chunk c of row r sits at c ^ (r % 8))
              ptx::st_shared_v4(prow + (((2 * k) ^ (r & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
              ptx::st_shared_v4(prow + (((2 * k + 1) ^ (r & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
            } else {
              ptx::tmem_st_x8(tS + 8 * k, pk);
            }
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int e = 32 * k + 2 * c;
              pk[c] = (DT == DT_BF16) ? ptx::pack_bf16x2(sv[e], sv[e + 1])
                                      : ptx::pack_f16x2(sv[e], sv[e + 1]);
            }
            ptx::tmem_st_x16(tS + 16 * k, pk);
          }
        }
        li += ((sum0 + sum1) + (sum2 + sum3)) * sum_scale;
        if constexpr (C::PSMEM) {
          if (any_rescale) {
            // P is already relative to the moved reference; O_s holds every
            // previous PV product once PV number p_cnt - 1 is done (it had the
            // whole exponential phase to finish). The S registers are dead:
            // O is read 64 columns at a time with both loads in flight.
            const int n = p_cnt - 1;
            ok = warp_wait_bar(bar(B_PFREEB + 2 * s + (n & 1)), (n >> 1) & 1, ctl);
            if (!ok) break;
            ptx::tc_fence_after();
            if constexpr (D == 64) {
              uint32_t oa[64];
              ptx::tmem_ld_x64(tO, oa);
#pragma unroll
              for (int c = 0; c < 64; c += 2) {
                float a0, a1;
                ptx::fma2(a0, a1, __uint_as_float(oa[c]), __uint_as_float(oa[c + 1]), alpha, alpha,
                          0.f, 0.f);
                oa[c] = __float_as_uint(a0);
                oa[c + 1] = __float_as_uint(a1);
              }
              ptx::tmem_st_x64(tO, oa);
            }
#pragma unroll 1
            for (int cb = 0; cb + 128 <= D; cb += 128) {
              uint32_t oa[64], ob[64];
              ptx::tmem_ld_x64_nowait(tO + cb, oa);
              ptx::tmem_ld_x64_nowait(tO + cb + 64, ob);
              ptx::tmem_ld_wait_x64x2(oa, ob);
#pragma unroll
              for (int c = 0; c < 64; c += 2) {
                float a0, a1, b0, b1;
                ptx::fma2(a0, a1, __uint_as_float(oa[c]), __uint_as_float(oa[c + 1]), alpha, alpha,
                          0.f, 0.f);
                ptx::fma2(b0, b1, __uint_as_float(ob[c]), __uint_as_float(ob[c + 1]), alpha, alpha,
                          0.f, 0.f);
                oa[c] = __float_as_uint(a0);
                oa[c + 1] = __float_as_uint(a1);
                ob[c] = __float_as_uint(b0);
                ob[c + 1] = __float_as_uint(b1);
              }
              ptx::tmem_st_x64(tO + cb, oa);
              ptx::tmem_st_x64(tO + cb + 64, ob);
            }
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        if constexpr (C::PSMEM) ptx::fence_proxy_async_smem();   // P visible to the MMA
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(C::PSMEM ? B_PFULLB + 2 * s + (p_cnt & 1) : B_PFULL + s));
        ++p_cnt;
        if constexpr (DT == DT_E4M3) {
          if (j + 1 < ns) {
            fp8_factors(kd_next, vd_next, cj_cur, bias_cur, ssc_cur);
            if (j + 2 < ns) {
              kd_next = __ldg(kd_row + U.j0 + j + 2);
              vd_next = __ldg(vd_row + U.j0 + j + 2);
            }
          }
        }
      }
      if (!ok) break;

      // ------------------------------------------------------------ epilogue
      ok = warp_wait_bar(bar(B_OFULL + s), u_it & 1, ctl);
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv = (DT == DT_E4M3 ? vref : 1.f) / li;
      const bool live = row < p.Nq;
      // l carries the factor 2^PSHIFT of the FP8 instance (0 otherwise)
      const float lse_row = (mi + ptx::lg2(li) - C::PSHIFT) * 0.6931471805599453f;
      if constexpr (SPLIT) {
        // split instances (few query rows, packed heads): one lane stores its row
        if (p.n_splits > 1) {
          // partial result of this key range: FP32 O / l and its LSE
          const long long prow = (((long long)U.sp * p.B + U.b) * p.Hq + hrow) * p.Nq + row;
          float* dst = p.o_part + prow * D;
#pragma unroll 1
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t o32[32];
            ptx::tmem_ld_x32(tO + cb, o32);
            if (live) {
              float4* d4 = reinterpret_cast<float4*>(dst + cb);
#pragma unroll
              for (int c = 0; c < 8; ++c)
                d4[c] = make_float4(__uint_as_float(o32[4 * c]) * inv, __uint_as_float(o32[4 * c + 1]) * inv,
                                    __uint_as_float(o32[4 * c + 2]) * inv,
                                    __uint_as_float(o32[4 * c + 3]) * inv);
            }
          }
          if (live) p.lse_part[prow] = lse_row;
        } else {
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                           (((long long)U.b * p.Nq + row) * p.Hq + hrow) * D;
#pragma unroll 1
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t o32[32];
            ptx::tmem_ld_x32(tO + cb, o32);
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float a = __uint_as_float(o32[2 * c]) * inv;
              const float b = __uint_as_float(o32[2 * c + 1]) * inv;
              pk[c] = (DT == DT_F16) ? ptx::pack_f16x2(a, b) : ptx::pack_bf16x2(a, b);
            }
            if (live) {
              uint4* d4 = reinterpret_cast<uint4*>(orow + cb);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                d4[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
          }
          if (live) p.lse[((long long)U.b * p.Hq + hrow) * p.Nq + row] = lse_row;
        }
      } else {
        // Full query tiles: a row-per-lane store would write 16 bytes into each
        // of 32 rows (32 cache lines) per instruction. After an 8 x 8 transpose
        // of 16-byte pieces inside each lane octet, lane 8g + i holds piece i of
        // the rows 8g .. 8g + 7 of this warp, so each store instruction writes
        // four whole 128-byte lines.
        const int rb = 32 * quarter + 8 * (lane >> 3);   // first tile row of this lane's octet
        const int pc = lane & 7;                          // 16-byte piece stored by this lane
        uint16_t* obase = reinterpret_cast<uint16_t*>(p.o);
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 64) {   // 64 columns = 128 bytes of a row
          uint32_t o64[64];
          ptx::tmem_ld_x64(tO + cb, o64);
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float a = __uint_as_float(o64[2 * c]) * inv;
            const float b = __uint_as_float(o64[2 * c + 1]) * inv;
            w[c] = (DT == DT_F16) ? ptx::pack_f16x2(a, b) : ptx::pack_bf16x2(a, b);
          }
          octet_transpose(w, lane);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int pos = m_s + rb + k;
            if (pos < p.Nq) {
              uint16_t* dst = obase + (((long long)U.b * p.Nq + pos) * p.Hq + hrow) * D + cb;
              reinterpret_cast<uint4*>(dst)[pc] =
                  make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
          }
        }
        if (live) p.lse[((long long)U.b * p.Hq + hrow) * p.Nq + row] = lse_row;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(B_OEMPTY + s));
      ++u_it;
    }
  } else {
    // idle warps of the MMA/TMA warpgroup
    if constexpr (QST == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
  }

  // --------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attn
