// attention.cuh -- joint (non-causal) flash attention on sm_103a tensor cores,
// BF16 and FP8 (E4M3) operands.
//
// Joint attention of "Speed up image generation with FLUX 3 Image Klein on
// NVIDIA Blackwell GPUs" (section "FLUX 3 inference with TensorRT LLM
// VisualGen"): every query token of [text | image | reference] attends to
// every key token of the same (batch, head); no mask.  The page measures the
// BF16 "VANILLA" attention at about 60 % of DiT kernel time and replaces it
// with FP8 attention (Q.K and P.V in FP8) in section "Quantized and sparse
// attention"; this kernel is that step in both precisions.
//
// One CTA = two 128-row query tiles (0 and 1) of one (b, h) that share every
// K/V tile.  Warp roles (Roles<>):
//   BF16 and Sol (352 threads):
//     warps 0-3  softmax + epilogue of query tile 0 (thread r owns row r, TMEM
//                lane r; the output tile leaves through shared memory and a
//                TMA store)
//     warps 4-7  softmax + epilogue of query tile 1
//     warp 8     TMA producer of the K ring
//     warp 9     TMEM allocator and tcgen05.mma issuer (one elected lane)
//     warp 10    TMA producer of both Q tiles and of the V ring
//   FP8, plain and with repair blocks (SPLIT, 640 threads):
//     warps 0-7 / 8-15  softmax + epilogue of tile 0 / 1: warp w takes 16 of
//                the 32 TMEM lanes of quadrant w % 4, two threads per row
//                (the even and the odd keys)
//     warp 16    K ring; warp 17 TMEM and the QK MMAs; warp 18 Q and the V
//                ring; warp 19 the P.V and row-sum MMAs
// TMEM (512 columns).  BF16 (and the repair blocks): S_0 at 0, S_1 at 128,
// O_0 at 256, O_1 at 384; the softmax of a tile overwrites its S with P, and
// the P.V MMA reads P straight from TMEM as its A operand.  FP8: one S region
// at 0 that the tiles take in turns, l_0 / l_1 at 128 / 160, P_0 / P_1 at
// 192 / 224, O as in BF16: P has its own columns, so the S region takes the
// next scores while the softmax still works on these, and the QK and P.V
// streams share no TMEM (which is what lets two warps issue them).
//
// BF16: the MMA issue order is  QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j)
// QK_1(j+1) | ...  so while the softmax of tile 0 works on S_0(j+1) the
// tensor core runs PV_1(j) and QK_1(j+1), and the other way round: each
// tile's softmax hides behind the other tile's two MMAs.  The
// MMAs of one thread complete in issue order, which is what makes two things
// safe: QK_t(j+1) overwrites the S_t columns that PV_t(j) reads P from, and
// the commit that signals S_t(j+1) also means that PV_t(j) has landed in O_t,
// so the softmax may rescale O_t as soon as it sees S_t(j+1).
//
// Online softmax in log2 units with a deferred rescale (BF16): the running
// max m only moves when a tile's max exceeds it by more than 2^8; until then
// p = 2^(s - m) may reach 2^8, which bf16 and the fp32 sums carry exactly as
// well.  O and l always use the same m, so the result is unchanged; most
// tiles then skip the O rescale (a TMEM round trip of 128 columns).  FP8
// rescales whenever m moves, because P is stored as E4M3 of 256 p <= 448.
//
// BF16: operands are bf16 (kind::f16, K = 16 per MMA).  A 128 x 128 tile is
// two 16 KB halves (head-dim columns 0-63, 64-127), each 128 rows x 128 bytes
// with the 128-byte TMA swizzle -- the canonical SW128 layout the MMA
// descriptors describe (K-major for Q and K; MN-major for V, read in place
// from [B, N, H, 128]).  P is bf16, two per TMEM column.
//
// FP8: Q', K' are E4M3 codes [B, H, N, 128] and V is E4M3 transposed
// [B, H, 128, Npad] (kind::f8f6f4, K = 32 per MMA; the keys of every 8 in
// the order 0 2 4 6 1 3 5 7, see SPLIT below).  A 128 x 128 tile is one
// 16 KB SW128 block, K-major for all three (for V^T the keys are the K
// dimension of P.V).  P is E4M3 of 256 p; the row sum l adds the values the
// codes stand for, so that O = sum p~ v / sum p~ is a convex combination of
// the V rows whatever the rounding of P.  Scores are scaled by s_q s_k and
// the output by s_v (per-(b, h) scales).  P stays in TMEM and the tensor
// core sums it (P times a tile of ones); the repair blocks of the VC instance
// sum their bf16 P in registers and hand the sum to the l column.
//
// VC-Attention repair (REP, FP8 only; vc_repair.cuh selects the tokens):
// the CTA first runs ceil(R / 128) repair blocks in BF16 -- K_rep = k' / s_k
// and V_rep = v / s_v of the R repaired key tokens, so that scores and P.V
// come out in the units of the E4M3 blocks -- and then the FP8 blocks over
// the N - R other keys (positions 0 .. N-R-1 of the codes).  The repair QK
// needs Q in bf16: the softmax warps convert their rows of the E4M3 Q tile
// (exact: every E4M3 value is a bf16 value) into the V ring's memory, which
// stays idle until the QK warp signals the last repair QK (qbf_free); the
// repair K and V tiles have their own 64 KB, which the E4M3 kernel has to
// spare, so the K ring fills from the start.  A repair block's S and P (bf16,
// over S) take per-tile columns as in the BF16 kernel; its row sum adds the
// fp32 p.
//
// Sol-Attention (SOL, BF16; sol_sparse.cuh builds the lists): the CTA walks
// only the key blocks in its list -- the union of the blocks its two query
// tiles keep -- and a tile that does not keep a block of the list writes
// P = 0 for it (its running max, sum and O stay as they are), so the MMA
// schedule stays the same for both tiles.
//
// Every wait is bounded (ptx.cuh); a wait that runs out sets the CTA abort
// flag and the error word, all roles stop issuing, drain what they issued,
// free TMEM and return.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace flux {
namespace attn {

constexpr int BM = 128;             // query rows per tile
constexpr int BN = 128;             // keys per tile
constexpr int HD = 128;             // head dim
constexpr int TILES = 2;            // query tiles per CTA
constexpr int CTA_ROWS = TILES * BM;
// Warp roles of an instance.  The BF16 and Sol instances run one softmax
// thread per row (4 warps per tile, 32x32b TMEM accesses) and one MMA issuer.
// The FP8 instances (SPLIT) run 8 warps per tile: warp w of a tile takes 16
// of the 32 TMEM lanes of quadrant w % 4 (16-lane TMEM shapes), and two
// threads share each row of the E4M3 blocks, one with the even and one with
// the odd key columns; two warps issue the MMAs, one the QKs and one the P.Vs
// and row sums (mma_split).  The FP8 MMAs take half the time of the BF16
// ones, and with one thread per row and one issuer the kernel ran at the
// pace of the softmax chains and of the issuer's barrier checks.
template <bool FP8, bool REP, bool SOL>
struct Roles {
  static constexpr bool SPLIT = FP8 && !SOL;
  static constexpr int SOFTMAX_WARPS = (SPLIT ? 8 : 4) * TILES;
  static constexpr int LOAD_K = SOFTMAX_WARPS;  // TMA producer of the K ring
  static constexpr int MMA = LOAD_K + 1;        // MMA issuer (SPLIT: of the QKs), TMEM owner
  static constexpr int LOAD_V = MMA + 1;        // TMA producer of Q and the V ring
  static constexpr int MMA_PV = LOAD_V + 1;     // SPLIT: issuer of the P.V and row-sum MMAs
  static constexpr int THREADS = 32 * (SPLIT ? MMA_PV + 1 : LOAD_V + 1);  // 352, SPLIT 640
  static constexpr int TILE_THREADS = 32 * SOFTMAX_WARPS / TILES;  // p_full / s_free arrivals per tile
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t HALF = BM * 128;  // one SW128 block: 128 rows x 128 bytes = 16 KB

__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }        // S_t / P_t
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; } // O_t
__host__ __device__ constexpr uint32_t col_l(int t) { return 128u + 32u * t; }  // FP8: l_t (16 columns used)
__host__ __device__ constexpr uint32_t col_p(int t) { return 192u + 32u * t; }  // FP8: P_t (E4M3)

// FP8 TMEM: the row sums l of the E4M3 blocks come from the tensor core (P
// times a tile of ones, into 16 columns per tile that O's rescale also
// scales), P_t lives in 32 columns (four E4M3 codes per column), and the two
// tiles take turns in one S region (col_s(0)) to make room for both.  The
// repair blocks (BF16, per-tile S columns, before the E4M3 blocks) keep their
// register sums, carried in l beside the column.

template <bool FP8>
struct Traits {
  static constexpr uint32_t TILE = FP8 ? HALF : 2 * HALF;  // bytes of one 128 x 128 operand tile
  // BF16: 2 K and 3 V stages measured ~1 % faster than 3 and 2 (same 160 KB)
  static constexpr int KST = FP8 ? 4 : 2;                  // K ring stages
  static constexpr int VST = FP8 ? 4 : 3;                  // V ring stages
  // How far (log2 units) a tile's max may exceed the running max before O
  // and l are rescaled: p = 2^(s - m) stays <= 2^RESCALE.
  static constexpr float RESCALE = FP8 ? 0.f : 8.f;
};

template <bool FP8>
struct __align__(1024) Smem {
  static constexpr uint32_t TILE = Traits<FP8>::TILE;
  static constexpr int KST = Traits<FP8>::KST;
  static constexpr int VST = Traits<FP8>::VST;
  uint8_t q[TILES][TILE];
  uint8_t k[KST][TILE];
  uint8_t v[VST][TILE];
  // FP8 only: the repair K and V tiles of VC-Attention (bf16, 32 KB each).  The
  // E4M3 rings leave this much of the SM's shared memory unused anyway (one
  // CTA per SM: TMEM holds one CTA's 512 columns).
  uint8_t rep[FP8 ? 2 : 1][FP8 ? 2 * HALF : 16];
  uint64_t q_full[TILES];
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[TILES], p_full[TILES], o_full[TILES];
  uint64_t s_free[TILES];              // FP8: tile t's S is in registers (128 arrivals)
  uint64_t o_done[TILES];              // FP8: PV_t of the last block has completed
  uint64_t qbf_full[TILES];            // REP: tile t's rows converted to bf16 (128 arrivals)
  uint64_t krep_full, krep_empty;      // REP: the repair K tile slot
  uint64_t vrep_full, vrep_empty;      // REP: the repair V tile slot
  uint64_t qbf_free;                   // REP: last repair QK of both tiles done
  uint64_t lrep_full[TILES];           // SPLIT REP without E4M3 blocks: the repair row sums are in TMEM
  uint64_t mma_drain;
  uint64_t mma_drain2;                 // SPLIT: the P.V issuer's own drain
  uint64_t never;  // nothing arrives here (forced-timeout debug path)
  uint32_t tmem_base;
  int abort;
};
template <bool FP8>
constexpr size_t smem_bytes() {
  return sizeof(Smem<FP8>) + 1024;  // + slack to align the base to 1024
}

struct Params {
  __nv_bfloat16* out;    // [B, N, H, 128]
  uint32_t* err;
  const float* scales;   // FP8: [B*H, 3] (s_q, s_k, s_v); BF16: unused
  int N, H, nkv;         // nkv: key blocks in all (repair blocks first)
  int nrep, rep_keys;    // REP: repair blocks and repaired keys R (0 otherwise)
  int main_keys;         // keys of the E4M3 / BF16 blocks: N - R
  const uint16_t* sol_list;  // SOL: [B*H][ncta][sol_nb] key block | tile keep bits << 14
  const int* sol_count;      // SOL: [B*H][ncta] entries of each list
  int sol_nb;
  float scale_log2;      // log2(e) / sqrt(128)
  int debug;
};

// Wait for a phase without looking at the abort flag (teardown drains only).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// Load one 128-row operand tile (rows `row0..+127` of slice `bh`) of a
// [.., rows, 128 elements] tensor map: two 64-column boxes for bf16, one
// 128-byte box for E4M3.  Rows past the end are zero-filled.
template <bool FP8>
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh) {
  tma_load_3d(dst, map, bar, 0, row0, bh);
  if (!FP8) tma_load_3d(dst + HALF, map, bar, 64, row0, bh);
}

// Drain a ring: the latest phase of every full-barrier a copy was issued on
// has completed (nothing may still be writing shared memory at exit).
template <int ST>
__device__ __forceinline__ void drain_ring(uint64_t (&full)[ST], int issued, uint32_t* err) {
  for (int s = 0; s < ST; ++s) {
    const int cnt = issued > s ? (issued - s + ST - 1) / ST : 0;
    if (cnt > 0) mbar_drain(&full[s], (cnt - 1) & 1, err);
  }
}

// REP shared memory: the two bf16 Q tiles in the V ring (32 KB each, idle
// until qbf_free), the repair K and V tiles in their own region, so that the
// K ring fills from the start.
template <bool FP8>
__device__ __forceinline__ uint8_t* qbf_tile(Smem<FP8>& sm, int t) {
  static_assert(!FP8 || sizeof(Smem<FP8>::v) >= TILES * 2 * HALF, "the bf16 Q tiles of the repair blocks live in the V ring");
  return &sm.v[0][0] + t * 2 * HALF;
}
template <bool FP8>
__device__ __forceinline__ uint8_t* krep_tile(Smem<FP8>& sm) { return &sm.rep[0][0]; }
template <bool FP8>
__device__ __forceinline__ uint8_t* vrep_tile(Smem<FP8>& sm) { return &sm.rep[FP8 ? 1 : 0][0]; }
// FP8: tile t's 16 KB staging half for its output (the second half is its Q
// tile) -- the repair K region, whose tile is consumed before the E4M3 blocks
// begin, and unused without repair blocks.
template <bool FP8>
__device__ __forceinline__ uint8_t* out_stage(Smem<FP8>& sm, int t) { return &sm.rep[0][0] + t * HALF; }
// FP8: 16 rows x 128 keys of E4M3 1.0 (0x38; 2 KB, every byte the same,
// so its swizzle does not matter) -- the repair V region, which the MMA
// thread fills once the last repair P.V has read it (or at once without
// repair blocks).
template <bool FP8>
__device__ __forceinline__ uint8_t* ones_tile(Smem<FP8>& sm) { return &sm.rep[FP8 ? 1 : 0][0]; }

// K ring producer: K_j into stage j % KST once both tiles' QK of its
// previous occupant have completed.  REP: the repair K tiles too (into their
// own slot, each once both tiles' QK of the one before it has completed),
// issued first.
template <bool FP8, bool REP, bool SOL>
__device__ __forceinline__ void load_k(Smem<FP8>& sm, const CUtensorMap* tk, const CUtensorMap* tkr, int bh,
                                       int nkv, int nrep, const uint16_t* lst, volatile int* ab, uint32_t* err) {
  constexpr uint32_t TILE = Traits<FP8>::TILE;
  constexpr int KST = Traits<FP8>::KST;
  int issued = 0;
  if (REP) {
    int rep_issued = 0;
    bool ok = true;
    for (int i = 0; i < nrep && ok; ++i) {
      if (i > 0 && !mbar_wait(&sm.krep_empty, (i - 1) & 1, ab, err)) { ok = false; break; }
      mbar_arrive_expect_tx(&sm.krep_full, 2 * HALF);
      load_rows<false>(smem_u32(krep_tile(sm)), tkr, &sm.krep_full, i * BN, bh);
      ++rep_issued;
    }
    if (!ok) {
      if (rep_issued > 0) mbar_drain(&sm.krep_full, (rep_issued - 1) & 1, err);
      return;
    }
    nkv -= nrep;
  }
  for (int j = 0; j < nkv; ++j) {
    const int kb = SOL ? (__ldg(lst + j) & 0x3FFF) : j;  // read before the wait
    const int ks = j % KST;
    const uint32_t ku = j / KST;
    if (ku > 0 && !mbar_wait(&sm.k_empty[ks], (ku - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.k_full[ks], TILE);
    load_rows<FP8>(smem_u32(sm.k[ks]), tk, &sm.k_full[ks], kb * BN, bh);
    ++issued;
  }
  drain_ring(sm.k_full, issued, err);
  if (REP && nrep > 0) mbar_drain(&sm.krep_full, (nrep - 1) & 1, err);
}

// Q and V ring producer: both Q tiles once, then V_j into stage j % VST once
// both tiles' PV of its previous occupant have completed.  REP: the repair V
// tiles first (into their own slot, each once both tiles' PV of the one
// before it has completed), and the ring only after qbf_free (it holds the
// bf16 Q tiles until the last repair QK).
template <bool FP8, bool REP, bool SOL>
__device__ __forceinline__ void load_qv(Smem<FP8>& sm, const CUtensorMap* tq, const CUtensorMap* tv,
                                        const CUtensorMap* tvr, int q0, int bh, int b, int h, int nkv, int nrep,
                                        const uint16_t* lst, volatile int* ab, uint32_t* err) {
  constexpr uint32_t TILE = Traits<FP8>::TILE;
  constexpr int VST = Traits<FP8>::VST;
#pragma unroll
  for (int t = 0; t < TILES; ++t) {
    mbar_arrive_expect_tx(&sm.q_full[t], TILE);
    load_rows<FP8>(smem_u32(sm.q[t]), tq, &sm.q_full[t], q0 + t * BM, bh);
  }
  int issued = 0;
  bool rep_ok = true;
  if (REP) {
    int rep_issued = 0;
    for (int i = 0; i < nrep && rep_ok; ++i) {
      if (i > 0 && !mbar_wait(&sm.vrep_empty, (i - 1) & 1, ab, err)) { rep_ok = false; break; }
      mbar_arrive_expect_tx(&sm.vrep_full, 2 * HALF);
      load_rows<false>(smem_u32(vrep_tile(sm)), tvr, &sm.vrep_full, i * BN, bh);
      ++rep_issued;
    }
    if (rep_issued > 0) mbar_drain(&sm.vrep_full, (rep_issued - 1) & 1, err);
    rep_ok = rep_ok && mbar_wait(&sm.qbf_free, 0, ab, err);
    nkv = rep_ok ? nkv - nrep : 0;
  }
  for (int j = 0; j < nkv; ++j) {
    const int kb = SOL ? (__ldg(lst + j) & 0x3FFF) : j;  // read before the wait
    const int vs = j % VST;
    const uint32_t vu = j / VST;
    if (vu > 0 && !mbar_wait(&sm.v_empty[vs], (vu - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.v_full[vs], TILE);
    if (FP8) {
      // V^T [B*H, 128, Npad]: keys kb*128.. are the inner (x) coordinate.
      tma_load_3d(smem_u32(sm.v[vs]), tv, &sm.v_full[vs], kb * BN, 0, bh);
    } else {
      // V [B, N, H, 128] in place: box (64 dims, 1 head, 128 keys, 1 batch).
      tma_load_4d(smem_u32(sm.v[vs]), tv, &sm.v_full[vs], 0, h, kb * BN, b);
      tma_load_4d(smem_u32(sm.v[vs]) + HALF, tv, &sm.v_full[vs], 64, h, kb * BN, b);
    }
    ++issued;
  }
#pragma unroll
  for (int t = 0; t < TILES; ++t) mbar_drain(&sm.q_full[t], 0, err);
  drain_ring(sm.v_full, issued, err);
}

// Matrix descriptors are built once per CTA: the start-address field
// (address >> 4, 14 bits) of a shared-memory tile never carries into the
// other fields, so the descriptor of an operand at byte offset `off` inside a
// tile is the tile's descriptor plus off >> 4.  That keeps the single issuing
// thread at one add per MMA, which matters: it shares its scheduler with two
// softmax warps and must issue an MMA every 64 cycles to keep up.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t off) { return d + (off >> 4); }

// S = Q K^T over the 128 head dims (qd, kd: SW128 K-major tile descriptors).
//   BF16: 8 MMAs of 128 x 128 x 16; step kk covers head dims 16kk..16kk+15:
//         half kk/4 of the tile, 32-byte offset (kk%4) inside the swizzle row.
//   FP8:  4 MMAs of 128 x 128 x 32; step kk is the 32-byte offset 32kk.
template <bool FP8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qd, uint64_t kd) {
  if (FP8) {
    constexpr uint32_t ID = idesc_e4m3(BM, BN, false);
#pragma unroll
    for (int kk = 0; kk < HD / 32; ++kk) mma_e4m3_ss(d_tmem, desc_at(qd, kk * 32), desc_at(kd, kk * 32), ID, kk > 0);
  } else {
    constexpr uint32_t ID = idesc_f16(BM, BN, false);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
      mma_f16_ss(d_tmem, desc_at(qd, off), desc_at(kd, off), ID, kk > 0);
    }
  }
}

// O (+)= P V over the 128 keys of a tile (vd: V tile descriptor).
//   BF16: 8 MMAs of 128 x 128 x 16; step kk covers keys 16kk..16kk+15: P
//         columns 8kk.. (two bf16 per column), V rows 16kk.. (16 rows x 128 B
//         = 2 KB); V is MN-major: LBO = the other 64 head dims (the other
//         half), SBO = next 8 keys.
//   FP8:  4 MMAs of 128 x 128 x 32; step kk covers keys 32kk..: P columns
//         8kk.. (four E4M3 per column), V^T K-major at byte offset 32kk.
template <bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t vd, bool accumulate) {
  if (FP8) {
    constexpr uint32_t ID = idesc_e4m3(BM, HD, false);
#pragma unroll
    for (int kk = 0; kk < BN / 32; ++kk)
      mma_e4m3_ts(o_tmem, p_tmem + kk * 8, desc_at(vd, kk * 32), ID, (accumulate || kk > 0) ? 1u : 0u);
  } else {
    constexpr uint32_t ID = idesc_f16(BM, HD, true);
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk)
      mma_f16_ts(o_tmem, p_tmem + kk * 8, desc_at(vd, kk * 2048), ID, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// l_t (+)= P_t 1: the row sums of P by the tensor core, N = 16 (16 equal
// columns; the softmax reads the first), 4 MMAs of 128 x 16 x 32 with P from
// TMEM (p_tmem) and the ones tile from shared memory (od).
__device__ __forceinline__ void issue_l_e4m3(uint32_t l_tmem, uint32_t p_tmem, uint64_t od, bool accumulate) {
  constexpr uint32_t ID = idesc_e4m3(BM, 16, false);
#pragma unroll
  for (int kk = 0; kk < BN / 32; ++kk)
    mma_e4m3_ts(l_tmem, p_tmem + kk * 8, desc_at(od, kk * 32), ID, (accumulate || kk > 0) ? 1u : 0u);
}

// BF16 main loop of the issuing thread, for both query tiles in one fixed
// order: QK_0(0) QK_1(0), then per block j
//   PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1)  [each pair after p_full_t(j)]
// Tile descriptors: K-major SW128 (SBO = 8 rows x 128 B) for Q and K,
// MN-major SW128 for V (LBO = the other 64 head dims).
// S_t and P_t share TMEM columns, so QK_t(j+1) follows PV_t(j) in this
// thread's issue order, and the commit that signals S_t(j+1) also means that
// PV_t(j) has landed in O_t.
__device__ __forceinline__ void mma_main_bf16(Smem<false>& sm, uint32_t tmem, int nkv, volatile int* ab,
                                              uint32_t* err) {
  constexpr uint32_t TILE = Traits<false>::TILE;
  constexpr int KST = Traits<false>::KST, VST = Traits<false>::VST;
  uint64_t qd[TILES];
#pragma unroll
  for (int t = 0; t < TILES; ++t) qd[t] = sdesc_sw128(smem_u32(sm.q[t]), 16, 1024);
  const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
  const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), HALF, 1024);
  if (!mbar_wait(&sm.k_full[0], 0, ab, err)) return;
#pragma unroll
  for (int t = 0; t < TILES; ++t) {
    if (!mbar_wait(&sm.q_full[t], 0, ab, err)) return;
    tc_fence_after_sync();
    issue_qk<false>(tmem + col_s(t), qd[t], kd0);
    mma_commit(&sm.s_full[t]);
  }
  mma_commit(&sm.k_empty[0]);
  for (int j = 0; j < nkv; ++j) {
    const int vs = j % VST;
    if (!mbar_wait(&sm.v_full[vs], (j / VST) & 1, ab, err)) return;
    const uint64_t vd = desc_at(vd0, vs * TILE);
    const int jn = j + 1;
    const int ks = jn % KST;
    const uint64_t kd = desc_at(kd0, ks * TILE);
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
      if (!mbar_wait(&sm.p_full[t], j & 1, ab, err)) return;
      tc_fence_after_sync();
      issue_pv<false>(tmem + col_o(t), tmem + col_s(t), vd, j > 0);
      if (t == TILES - 1) mma_commit(&sm.v_empty[vs]);
      if (jn < nkv) {
        if (t == 0) {
          if (!mbar_wait(&sm.k_full[ks], (jn / KST) & 1, ab, err)) return;
          tc_fence_after_sync();
        }
        // In issue order after PV_t(j), which read P_t from these columns.
        issue_qk<false>(tmem + col_s(t), qd[t], kd);
        mma_commit(&sm.s_full[t]);
        if (t == TILES - 1) mma_commit(&sm.k_empty[ks]);
      } else {
        mma_commit(&sm.o_full[t]);
      }
    }
  }
}

// The MMA issuer of the BF16 and Sol instances (the whole warp runs the
// loop, one elected lane issues: ptx.cuh), for both tiles.
__device__ __forceinline__ void mma_issuer(Smem<false>& sm, uint32_t tmem, int nkv, volatile int* ab, uint32_t* err) {
  if (nkv <= 0) {
#pragma unroll
    for (int t = 0; t < TILES; ++t) mma_commit(&sm.o_full[t]);
  } else {
    mma_main_bf16(sm, tmem, nkv, ab, err);
  }
  // Drain every MMA this thread issued before TMEM is released.
  mma_commit(&sm.mma_drain);
  mbar_drain(&sm.mma_drain, 0, err);
}

// SPLIT: the MMAs come from two warps.  A single issuing thread spent each
// block on six barrier checks in a row between its MMA groups, and the
// tensor pipe drained meanwhile (a per-block trace: ~1200 of ~2480 cycles).
// The QK and the P.V streams touch disjoint TMEM (the S region; O, l and P),
// and each has its own barriers, so one warp issues the QKs and another the
// P.V and row-sum MMAs: one's waits overlap the other's issue.  A commit
// tracks the MMAs of its own thread, which is all each barrier needs.
//
// QK warp, per block j: QK_1(j) after s_free_0(j), QK_0(j+1) after
// s_free_1(j) (both tiles' scores go through the one S region in turns).
// REP: first the repair QKs (bf16 Q from the converted tiles, K from the
// repair slot) into S_t per tile, each after the repair P.V that read the P
// over its columns (o_done_t); the E4M3 blocks begin once the last repair
// P.V of both tiles is done (their S, P and l columns overlap the repair S).
// nkv: the E4M3 blocks.
template <bool REP>
__device__ __forceinline__ void mma_qk_split(Smem<true>& sm, uint32_t tmem, int nkv, int nrep, volatile int* ab,
                                             uint32_t* err) {
  constexpr uint32_t TILE = Traits<true>::TILE;
  constexpr int KST = Traits<true>::KST;
  if constexpr (REP) {
    uint64_t qbd[TILES];
#pragma unroll
    for (int t = 0; t < TILES; ++t) qbd[t] = sdesc_sw128(smem_u32(qbf_tile(sm, t)), 16, 1024);
    const uint64_t krd = sdesc_sw128(smem_u32(krep_tile(sm)), 16, 1024);
    for (int i = 0; i < nrep; ++i) {
      if (!mbar_wait(&sm.krep_full, i & 1, ab, err)) return;
#pragma unroll
      for (int t = 0; t < TILES; ++t) {
        if (!mbar_wait(i == 0 ? &sm.qbf_full[t] : &sm.o_done[t], i == 0 ? 0 : (i - 1) & 1, ab, err)) return;
        tc_fence_after_sync();
        issue_qk<false>(tmem + col_s(t), qbd[t], krd);
        mma_commit(&sm.s_full[t]);
      }
      mma_commit(&sm.krep_empty);
      if (i == nrep - 1) mma_commit(&sm.qbf_free);
    }
    if (nkv <= 0) return;
    if (nrep > 0) {
#pragma unroll
      for (int t = 0; t < TILES; ++t)
        if (!mbar_wait(&sm.o_done[t], (nrep - 1) & 1, ab, err)) return;
    }
  }
  uint64_t qd[TILES];
#pragma unroll
  for (int t = 0; t < TILES; ++t) qd[t] = sdesc_sw128(smem_u32(sm.q[t]), 16, 1024);
  const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
  const uint32_t s_tmem = tmem + col_s(0);
  if (!mbar_wait(&sm.k_full[0], 0, ab, err)) return;
  if (!mbar_wait(&sm.q_full[0], 0, ab, err)) return;
  tc_fence_after_sync();
  issue_qk<true>(s_tmem, qd[0], kd0);
  mma_commit(&sm.s_full[0]);
  for (int j = 0; j < nkv; ++j) {
    const int ks = j % KST;
    if (j == 0 && !mbar_wait(&sm.q_full[1], 0, ab, err)) return;
    if (!mbar_wait(&sm.s_free[0], j & 1, ab, err)) return;
    tc_fence_after_sync();
    issue_qk<true>(s_tmem, qd[1], desc_at(kd0, ks * TILE));
    mma_commit(&sm.s_full[1]);
    mma_commit(&sm.k_empty[ks]);
    if (j + 1 < nkv) {
      const int kn = (j + 1) % KST;
      if (!mbar_wait(&sm.k_full[kn], ((j + 1) / KST) & 1, ab, err)) return;
      if (!mbar_wait(&sm.s_free[1], j & 1, ab, err)) return;
      tc_fence_after_sync();
      issue_qk<true>(s_tmem, qd[0], desc_at(kd0, kn * TILE));
      mma_commit(&sm.s_full[0]);
    }
  }
}

// P.V warp, per block j: PV_t(j) and l_t += P_t 1 after p_full_t(j), for
// t = 0, 1 (V_j must be in); o_done_t, then v_empty and, after the last
// block, o_full_t.  REP: first the repair P.Vs (bf16 P over S_t, V from the
// repair slot), each committed on o_done_t; the ones tile then takes the
// repair V slot, and the E4M3 P.V and row sums accumulate onto the repair
// blocks' O and the l the softmax put in its column.  nkv: the E4M3 blocks.
template <bool REP>
__device__ __forceinline__ void mma_pv_split(Smem<true>& sm, uint32_t tmem, int nkv, int nrep, volatile int* ab,
                                             uint32_t* err) {
  if constexpr (REP) {
    const uint64_t vrd = sdesc_sw128(smem_u32(vrep_tile(sm)), HALF, 1024);
    for (int i = 0; i < nrep; ++i) {
      if (!mbar_wait(&sm.vrep_full, i & 1, ab, err)) return;
#pragma unroll
      for (int t = 0; t < TILES; ++t) {
        if (!mbar_wait(&sm.p_full[t], i & 1, ab, err)) return;
        tc_fence_after_sync();
        issue_pv<false>(tmem + col_o(t), tmem + col_s(t), vrd, i > 0);
        mma_commit(&sm.o_done[t]);
        if (nkv <= 0 && i == nrep - 1) mma_commit(&sm.o_full[t]);
      }
      mma_commit(&sm.vrep_empty);
    }
    if (nkv <= 0) return;
    if (nrep > 0 && !mbar_wait(&sm.vrep_empty, (nrep - 1) & 1, ab, err)) return;  // V_rep read, the slot is free
  }
  const int ph = REP ? nrep : 0;  // p_full phases after the repair blocks
  {  // the ones tile of the row sums, 64 bytes per lane
    uint4* o = reinterpret_cast<uint4*>(ones_tile(sm)) + (threadIdx.x & 31) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
    __syncwarp();
  }
  constexpr uint32_t TILE = Traits<true>::TILE;
  constexpr int VST = Traits<true>::VST;
  const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
  const uint64_t od = sdesc_sw128(smem_u32(ones_tile(sm)), 16, 1024);
  for (int j = 0; j < nkv; ++j) {
    const int vs = j % VST;
    if (!mbar_wait(&sm.v_full[vs], (j / VST) & 1, ab, err)) return;
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
      if (!mbar_wait(&sm.p_full[t], (j + ph) & 1, ab, err)) return;
      tc_fence_after_sync();
      issue_pv<true>(tmem + col_o(t), tmem + col_p(t), desc_at(vd0, vs * TILE), REP || j > 0);
      issue_l_e4m3(tmem + col_l(t), tmem + col_p(t), od, REP || j > 0);
      mma_commit(&sm.o_done[t]);
      if (j == nkv - 1) mma_commit(&sm.o_full[t]);
    }
    mma_commit(&sm.v_empty[vs]);
  }
}

// Either SPLIT issuer, then the drain of its own MMAs (before TMEM goes).
// nkv: all key blocks (REP: nrep repair blocks first).
template <bool REP, bool QK>
__device__ __forceinline__ void mma_split(Smem<true>& sm, uint32_t tmem, int nkv, int nrep, volatile int* ab,
                                          uint32_t* err) {
  if (!REP) nrep = 0;
  if (QK) mma_qk_split<REP>(sm, tmem, nkv - nrep, nrep, ab, err);
  else mma_pv_split<REP>(sm, tmem, nkv - nrep, nrep, ab, err);
  uint64_t* drain = QK ? &sm.mma_drain : &sm.mma_drain2;
  mma_commit(drain);
  mbar_drain(drain, 0, err);
}

// Two E4M3 codes (round to nearest even, saturating) of a float pair, a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// The values two E4M3 codes stand for, exact in f16.
__device__ __forceinline__ __half2 e4m3x2_value(uint32_t c) {
  return __half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c), __NV_E4M3));
}

// REP: thread r converts row r of the E4M3 Q tile t into the bf16 tile the
// repair QK reads (both in the 128-byte-swizzled layout: a row's 16-byte
// chunk c sits at chunk position c ^ (r % 8); the bf16 tile is two halves of
// 64 head dims).  E4M3 values are exact in f16 and in bf16.
// NC chunks from chunk c0 on (SPLIT: the two warps of a TMEM quadrant take
// half a row each).
template <bool FP8, int NC = 8>
__device__ __forceinline__ void convert_q_row(Smem<FP8>& sm, int t, int r, int c0 = 0) {
  const uint8_t* src = sm.q[t] + r * 128;
  uint8_t* dst = qbf_tile(sm, t);
#pragma unroll
  for (int cc = 0; cc < NC; ++cc) {  // 16 codes: head dims 16c .. 16c + 15
    const int c = c0 + cc;
    const uint4 u = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = __half22float2(e4m3x2_value(wd[i] & 0xFFFFu));
      const float2 hi = __half22float2(e4m3x2_value(wd[i] >> 16));
      o[2 * i] = pack_bf16x2(lo.x, lo.y);
      o[2 * i + 1] = pack_bf16x2(hi.x, hi.y);
    }
    // dims 16c .. 16c+7 and 16c+8 .. 16c+15: half (16c) / 64, chunks 2 (c % 4) and 2 (c % 4) + 1
    uint8_t* row = dst + (c >> 2) * HALF + r * 128;
    const int k0 = 2 * (c & 3);
    *reinterpret_cast<uint4*>(row + ((k0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(row + (((k0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Max of a thread's NS scores: four chains of three-input max (eight chains
// measured 1 % slower in BF16 at N = 4608, the same in FP8).
constexpr int kMaxChains = 4;
template <int NS>
__device__ __forceinline__ float row_max(const uint32_t (&s)[NS]) {
  float acc[kMaxChains];
#pragma unroll
  for (int c = 0; c < kMaxChains; ++c) acc[c] = fmaxf(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]));
#pragma unroll
  for (int i = 2 * kMaxChains; i < NS; i += 2 * kMaxChains) {
#pragma unroll
    for (int c = 0; c < kMaxChains; ++c)
      acc[c] = fmax3(acc[c], __uint_as_float(s[i + 2 * c]), __uint_as_float(s[i + 2 * c + 1]));
  }
#pragma unroll
  for (int w = kMaxChains; w > 1; w /= 2) {
#pragma unroll
    for (int c = 0; c < w / 2; ++c) acc[c] = fmaxf(acc[c], acc[c + w / 2]);
  }
  return acc[0];
}

// One key block of the online softmax of query tile t of the BF16 and Sol
// instances (128 threads, thread r = row r): wait for S, mask the keys >=
// valid, update the running max m (log2 units) and sum l, write P over S
// (bf16, two per TMEM column), rescale O when the max moved (has_o: O already
// holds earlier blocks), and hand P to the MMA thread.  Returns false when
// the CTA gave up.
__device__ __forceinline__ bool softmax_block(Smem<false>& sm, int t, uint32_t s_addr, uint32_t o_addr,
                                              uint32_t phase, int valid, bool has_o, float sl2, float& m, float& l,
                                              volatile int* ab, uint32_t* err, bool keep = true) {
  constexpr float kRescale = Traits<false>::RESCALE;
  const bool ok = mbar_wait(&sm.s_full[t], phase, ab, err);
  if (__any_sync(0xFFFFFFFFu, !ok)) return false;
  tc_fence_after_sync();
  if (!keep) {  // SOL: the tile does not attend to this block: P = 0 (warp-uniform)
    uint32_t z[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) z[i] = 0u;
    tmem_st64(s_addr, z);
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(&sm.p_full[t]);
    return true;
  }
  uint32_t s[BN];
  tmem_ld128(s_addr, s);
  tmem_ld_wait(s);
  if (valid < BN) {
#pragma unroll
    for (int i = 0; i < BN; ++i)
      if (i >= valid) s[i] = __float_as_uint(-INFINITY);
  }
  // Row max: four independent chains of three-input max (depth 16, not 127).
  const float mx = row_max(s);
  const float m_tile = fmaxf(m, mx * sl2);
  // One decision per warp (TMEM moves are warp-wide); each row keeps its own alpha.
  const bool rescale = __any_sync(0xFFFFFFFFu, m_tile > m + kRescale);
  const float m_new = rescale ? m_tile : m;
  const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;  // 0 on the first tile
  const float nm = -m_new;
  // p = 2^(s sl2 - m): the argument of two scores per packed FMA; the row
  // sum in four packed accumulators.
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  {
    uint32_t pk[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) {
      float x0, x1;
      fma2(x0, x1, __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]), sl2, sl2, nm, nm);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      add2(sum[2 * (i & 3)], sum[2 * (i & 3) + 1], p0, p1);
      pk[i] = pack_bf16x2(p0, p1);
    }
    tmem_st64(s_addr, pk);
  }
  add2(sum[0], sum[1], sum[2], sum[3]);
  add2(sum[4], sum[5], sum[6], sum[7]);
  add2(sum[0], sum[1], sum[4], sum[5]);
  l = l * alpha + (sum[0] + sum[1]);
  // O_t holds the earlier blocks' P V already (see the issue order), and
  // nothing else writes it until this thread arrives on p_full below.
  if (rescale && has_o) {
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(o_addr + c * 32, o);
      tmem_ld_wait(o);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
      tmem_st32(o_addr + c * 32, o);
    }
  }
  tmem_st_wait();
  m = m_new;
  tc_fence_before_sync();
  mbar_arrive(&sm.p_full[t]);
  return true;
}

// Softmax and epilogue of query tile `t` of the BF16 and Sol instances (128
// threads, thread r = row r).
template <bool SOL>
__device__ __forceinline__ void softmax_epilogue(Smem<false>& sm, uint32_t tmem, const Params& prm, int b, int h,
                                                 int row0, int t, int nkv, const uint16_t* lst, volatile int* ab,
                                                 const CUtensorMap* tm_o) {
  const int r = threadIdx.x & (BM - 1);
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;  // TMEM lanes of this warp
  const uint32_t s_addr = tmem + lane_base + col_s(t);
  const uint32_t o_addr = tmem + lane_base + col_o(t);
  const float sl2 = prm.scale_log2;
  float m = -INFINITY;  // running max, in log2 units
  float l = 0.f;        // running row sum
  bool ok = true;
  if (SOL) {
    // list entry j: key block (14 bits) and the keep bits of the two tiles; a
    // block the tile skips still gets its (zero) P, so O is written from j = 0
    for (int j = 0; j < nkv && ok; ++j) {
      const uint32_t e = __ldg(lst + j);
      ok = softmax_block(sm, t, s_addr, o_addr, j & 1, prm.N - static_cast<int>(e & 0x3FFFu) * BN, j > 0, sl2, m,
                         l, ab, prm.err, (e >> (14 + t)) & 1u);
    }
  } else {
    for (int j = 0; j < nkv && ok; ++j)
      ok = softmax_block(sm, t, s_addr, o_addr, j & 1, prm.main_keys - j * BN, j > 0, sl2, m, l, ab, prm.err);
  }
  if (ok) {
    ok = mbar_wait(&sm.o_full[t], 0, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
  }
  if (!ok) return;
  tc_fence_after_sync();
  const float inv_l = 1.f / l;
  // O tile (bf16, 32 KB) -> the tile's own 32 KB Q buffer, which no MMA or
  // copy touches any more (its last QK completed before the PV that
  // signalled o_full), in the SW128 layout of the out tensor map: half c / 2
  // holds head dims 64 (c / 2) .., row r at byte 128 r, its 16-byte chunk k
  // at position k ^ (r % 8).  Then one thread writes the two halves with TMA
  // stores, which also clip rows >= N: whole 128-byte rows instead of each
  // thread's 16-byte pieces of rows H x 256 bytes apart.
  uint8_t* stage[2] = {sm.q[t], sm.q[t] + HALF};
#pragma unroll
  for (int c = 0; c < HD / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(o_addr + c * 32, o);
    tmem_ld_wait(o);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
    const int half = c >> 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = (c & 1) * 4 + i;  // 16-byte chunk within the 128-byte row of this half
      *reinterpret_cast<uint4*>(stage[half] + r * 128 + ((k ^ (r & 7)) << 4)) =
          make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
  fence_proxy_async_smem();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(BM) : "memory");
  if (r == 0) {
    tma_store_4d(tm_o, smem_u32(stage[0]), 0, h, row0, b);  // rows >= N are clipped
    tma_store_4d(tm_o, smem_u32(stage[1]), 64, h, row0, b);
    bulk_commit();
    bulk_wait_read_all();  // the staging buffer may go; the writes complete with the grid
  }
}

// ---------------------------------------------------------------- SPLIT FP8
// The FP8 instances with two threads per row (Roles::SPLIT).  Thread i
// of a warp owns lane (i / 4 + 8 (i % 2)) of the warp's 16 TMEM lanes and the
// key columns of parity (i / 2) % 2: its 64 scores of a block are keys
// 2k + par, k = 0..63 (16x64b loads).  The row max takes one shuffle with the
// partner thread (i ^ 2).  Its P codes go out with the same shape: register
// k' is P column 2k' + par, whose four bytes the P.V MMA takes as keys
// 4 (2k' + par) + b -- the thread puts there the codes of its scores 4k' + b,
// keys 8k' + 2b + par.  So within every 8 keys the MMA's K order is the key
// order 0, 2, 4, 6, 1, 3, 5, 7, and V^T is stored in that order
// (fp8_vt_kernel<true>); S, the masking and the row sums see keys in order.

struct SplitLanes {
  uint32_t s, o, l, p;  // TMEM addresses of this warp's 16 lanes (S, O_t, l_t, P_t)
  int par;              // key / column parity of this thread
};

// One key block of the online softmax of tile t for one SPLIT warp: wait for
// S, mask keys >= valid, max (with the partner thread), exp2 into E4M3 codes,
// wait for the previous P.V (it read P and wrote O, l), store P, rescale O
// and l when the max moved, hand P to the MMA thread.
//
// REP: the E4M3 blocks after nrep repair blocks: O holds their P.V from the
// start, their o_done phases come first, and at the first E4M3 block the
// thread puts the repair blocks' row sum l_rep (scaled like O) into its l
// column, which the row-sum MMAs then add to.
template <bool REP>
__device__ __forceinline__ bool softmax_block_split(Smem<true>& sm, int t, const SplitLanes& a, uint32_t phase,
                                                    int jm, int valid, float sl2, float& m, volatile int* ab,
                                                    uint32_t* err, int nrep = 0, float l_rep = 0.f) {
  constexpr float kPBias = 8.f;  // P = E4M3 of 256 p: folded into the exponent, cancels against l
  bool ok = mbar_wait(&sm.s_full[t], phase, ab, err);
  if (__any_sync(0xFFFFFFFFu, !ok)) return false;
  tc_fence_after_sync();
  uint32_t s[BN / 2];
  tmem_ld16x64(a.s, s);
  tmem_ld_wait(s);
  tc_fence_before_sync();
  mbar_arrive(&sm.s_free[t]);  // the S region may take the next QK now
  if (valid < BN) {
#pragma unroll
    for (int k = 0; k < BN / 2; ++k)
      if (2 * k + a.par >= valid) s[k] = __float_as_uint(-INFINITY);
  }
  float mx = row_max(s);
  mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));  // the row's other half
  const float m_tile = fmaxf(m, mx * sl2);
  // one decision per warp (TMEM moves are warp-wide); P = E4M3 of 256 p needs
  // the exact running max, so any rise rescales
  const bool rescale = __any_sync(0xFFFFFFFFu, m_tile > m);
  const float m_new = rescale ? m_tile : m;
  const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;  // 0 on the first block
  const float nm = kPBias - m_new;
  uint32_t pk[BN / 8];
#pragma unroll
  for (int i = 0; i < BN / 8; ++i) {
    float x0, x1, x2, x3;
    fma2(x0, x1, __uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1]), sl2, sl2, nm, nm);
    fma2(x2, x3, __uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3]), sl2, sl2, nm, nm);
    pk[i] = e4m3x2(ex2_approx(x0), ex2_approx(x1)) | (e4m3x2(ex2_approx(x2), ex2_approx(x3)) << 16);
  }
  if (jm > 0) {
    ok = mbar_wait(&sm.o_done[t], (REP ? jm - 1 + nrep : jm - 1) & 1, ab, err);
    if (__any_sync(0xFFFFFFFFu, !ok)) return false;
    tc_fence_after_sync();
  }
  tmem_st16x16(a.p, pk);  // waited for (tcgen05.wait::st) before p_full below
  const bool has_o = REP ? (jm > 0 || nrep > 0) : jm > 0;
  if (rescale && has_o) {
    // this thread's 64 of the row's O columns, and its l column (the row sum
    // MMA writes 16 equal columns; the pair keeps columns 0 and 1 scaled)
    const bool l_in_tmem = !REP || jm > 0;
    uint32_t o[HD / 2];
    tmem_ld16x64(a.o, o);
    uint32_t lv = 0;
    if (l_in_tmem) lv = tmem_ld16x1(a.l);
    tmem_ld_wait(o);
#pragma unroll
    for (int i = 0; i < HD / 2; i += 2) {
      float a0, a1;
      mul2(a0, a1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
      o[i] = __float_as_uint(a0);
      o[i + 1] = __float_as_uint(a1);
    }
    tmem_st16x64(a.o, o);
    if (l_in_tmem) {
      tmem_ld_wait(lv);
      tmem_st16x1(a.l, __float_as_uint(__uint_as_float(lv) * alpha));
    }
  }
  if (REP && jm == 0 && nrep > 0) tmem_st16x1(a.l, __float_as_uint(l_rep * alpha));
  tmem_st_wait();
  m = m_new;
  tc_fence_before_sync();
  mbar_arrive(&sm.p_full[t]);
  return true;
}

// The repair blocks (bf16 P) of the SPLIT repair instance: thread i of a warp
// holds rows g = i / 4 and g + 8 of the warp's 16 TMEM lanes and, of each
// row, the keys 8k + 2q and 8k + 2q + 1 (q = i % 4, k = 0..15): a 16x256b load
// of S puts row g + 8h, key 8k + 2q + e in register 4k + 2h + e.  P is bf16
// with keys 2c and 2c + 1 in column c, so the thread's P is exactly columns
// 4k + q of its two rows, which a 16x128b store writes (register 2k + h) over
// S: no exchange between threads and no change of key order.  The row max
// takes two shuffles over the four threads of a row; each thread keeps its
// part of the row sums.  Row g + 8 (i % 2) is the thread's row in the 16x64b
// layout of the E4M3 blocks that follow.
__device__ __forceinline__ float max32_of_row(const uint32_t (&s)[BN / 2], int hr) {
  float acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = fmaxf(__uint_as_float(s[4 * c + 2 * hr]), __uint_as_float(s[4 * c + 2 * hr + 1]));
#pragma unroll
  for (int k = 4; k < 16; k += 4) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      acc[c] = fmax3(acc[c], __uint_as_float(s[4 * (k + c) + 2 * hr]), __uint_as_float(s[4 * (k + c) + 2 * hr + 1]));
  }
  return fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3]));
}

template <bool FP8>
__device__ __forceinline__ bool softmax_block_b16s(Smem<FP8>& sm, int t, const SplitLanes& a, uint32_t phase,
                                                   int jm, int valid, float sl2, float (&m)[2], float (&l)[2],
                                                   volatile int* ab, uint32_t* err) {
  // FP8: the scale of the E4M3 blocks (P of 256 p, 2^8 folded into the exponent)
  constexpr float kPBias = FP8 ? 8.f : 0.f;
  constexpr float kRescale = Traits<FP8>::RESCALE;
  bool ok = mbar_wait(&sm.s_full[t], phase, ab, err);
  if (__any_sync(0xFFFFFFFFu, !ok)) return false;
  tc_fence_after_sync();
  uint32_t s[BN / 2];
  tmem_ld16x256(a.s, s);
  tmem_ld_wait(s);
  const int k0 = 2 * a.par;    // par = q here: the thread's first key of every 8
  if (valid < BN) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (8 * k + k0 + e >= valid) s[4 * k + 2 * h2 + e] = __float_as_uint(-INFINITY);
  }
  float mt[2], mn[2], alpha[2], nm[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    float mx = max32_of_row(s, hr);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    mt[hr] = fmaxf(m[hr], mx * sl2);
  }
  const bool rescale = __any_sync(0xFFFFFFFFu, mt[0] > m[0] + kRescale || mt[1] > m[1] + kRescale);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    mn[hr] = rescale ? mt[hr] : m[hr];
    alpha[hr] = rescale ? ex2_approx(m[hr] - mn[hr]) : 1.f;  // 0 on the first block
    nm[hr] = kPBias - mn[hr];
  }
  uint32_t pk[BN / 4];
  float sum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float x0, x1;
      fma2(x0, x1, __uint_as_float(s[4 * k + 2 * hr]), __uint_as_float(s[4 * k + 2 * hr + 1]), sl2, sl2, nm[hr],
           nm[hr]);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      add2(sum[hr][0], sum[hr][1], p0, p1);
      pk[2 * k + hr] = pack_bf16x2(p0, p1);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) l[hr] = l[hr] * alpha[hr] + (sum[hr][0] + sum[hr][1]);
  // P over S_t (bf16, the first 64 of its 128 columns): PV_t(j-1) has read
  // the previous P and landed in O_t -- the QK warp waits for its commit
  // before QK_t(j), whose commit signalled S_t(j)
  tmem_st16x128(a.p, pk);
  if (rescale && jm > 0) {
    uint32_t o[HD / 2];
    tmem_ld16x256(a.o, o);
    tmem_ld_wait(o);
#pragma unroll
    for (int k = 0; k < 16; ++k)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float a0, a1;
        mul2(a0, a1, __uint_as_float(o[4 * k + 2 * hr]), __uint_as_float(o[4 * k + 2 * hr + 1]), alpha[hr],
             alpha[hr]);
        o[4 * k + 2 * hr] = __float_as_uint(a0);
        o[4 * k + 2 * hr + 1] = __float_as_uint(a1);
      }
    tmem_st16x256(a.o, o);
  }
  tmem_st_wait();
  m[0] = mn[0];
  m[1] = mn[1];
  tc_fence_before_sync();
  mbar_arrive(&sm.p_full[t]);
  return true;
}

// Softmax and epilogue of query tile t for one SPLIT warp (8 per tile).  The
// epilogue switches to whole rows: the two warps of a TMEM quadrant read its
// 32 lanes with 32x32b loads, warp half hh taking O columns 64 hh .. +63,
// which is output half hh of the tile (head dims 64 hh ..).
// REP: first the Q conversion (each warp of a quadrant half a row) and the
// repair blocks in the 16x256b layout; their running max and row sum carry
// over to the E4M3 blocks (the thread's row there is its row i % 2 of them).
template <bool REP>
__device__ __forceinline__ void softmax_epilogue_split(Smem<true>& sm, uint32_t tmem, const Params& prm, int b,
                                                       int h, int row0, int t, int nkv, volatile int* ab,
                                                       const CUtensorMap* tm_o) {
  const int wt = (threadIdx.x >> 5) & 7;  // warp within the tile
  const int qd = wt & 3;                  // TMEM lane quadrant (= warp % 4)
  const int hh = wt >> 2;                 // which 16 lanes of the quadrant; later, which output half
  const int i = threadIdx.x & 31;
  SplitLanes a;
  const uint32_t lanes16 = static_cast<uint32_t>(32 * qd + 16 * hh) << 16;
  a.s = tmem + lanes16 + col_s(0);
  a.o = tmem + lanes16 + col_o(t);
  a.l = tmem + lanes16 + col_l(t);
  a.p = tmem + lanes16 + col_p(t);
  a.par = (i >> 1) & 1;
  const float* sc = prm.scales + 3 * (static_cast<size_t>(b) * prm.H + h);
  const float sl2 = prm.scale_log2 * __ldg(sc) * __ldg(sc + 1);
  const float out_scale = __ldg(sc + 2);
  const int nrep = REP ? prm.nrep : 0;
  const int nmain = nkv - nrep;
  float m = -INFINITY;  // running max of this thread's row, log2 units
  float l_rep = 0.f;    // REP: the repair blocks' row sum of that row
  bool ok = true;
  if (REP && nrep > 0) {
    ok = mbar_wait(&sm.q_full[t], 0, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) return;
    convert_q_row<true, 4>(sm, t, 32 * qd + i, 4 * hh);
    fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
    mbar_arrive(&sm.qbf_full[t]);
    SplitLanes ar = a;
    ar.s = tmem + lanes16 + col_s(t);  // S_t and P over it, per tile
    ar.p = ar.s;
    ar.par = i & 3;
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
    for (int k = 0; k < nrep && ok; ++k)
      ok = softmax_block_b16s<true>(sm, t, ar, k & 1, k, prm.rep_keys - k * BN, sl2, m2, l2, ab, prm.err);
    if (!ok) return;
    float lt[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      lt[hr] = l2[hr] + __shfl_xor_sync(0xFFFFFFFFu, l2[hr], 1);
      lt[hr] += __shfl_xor_sync(0xFFFFFFFFu, lt[hr], 2);
    }
    m = (i & 1) ? m2[1] : m2[0];
    l_rep = (i & 1) ? lt[1] : lt[0];
  }
  for (int j = 0; j < nmain && ok; ++j)
    ok = softmax_block_split<REP>(sm, t, a, (j + nrep) & 1, j, prm.main_keys - j * BN, sl2, m, ab, prm.err, nrep,
                                  l_rep);
  if (ok) {
    ok = mbar_wait(&sm.o_full[t], 0, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
  }
  if (REP && ok && nmain == 0) {
    // no E4M3 block: the repair sums go into the l column for the epilogue,
    // once every P.V is done (the other tile's repair P spans these columns)
    ok = mbar_wait(&sm.o_full[1 - t], 0, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
    if (ok) {
      tc_fence_after_sync();
      tmem_st16x1(a.l, __float_as_uint(l_rep));
      tmem_st_wait();
      tc_fence_before_sync();
      // the two warps of a quadrant wrote one half of its lanes each
      mbar_arrive(&sm.lrep_full[t]);
      ok = mbar_wait(&sm.lrep_full[t], 0, ab, prm.err);
      if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
    }
  }
  if (!ok) return;
  tc_fence_after_sync();
  const int r = 32 * qd + i;  // row of the tile for the epilogue
  const uint32_t lanes32 = static_cast<uint32_t>(32 * qd) << 16;
  uint32_t lv = tmem_ld1(tmem + lanes32 + col_l(t));  // the tensor core's row sum (column 0)
  tmem_ld_wait(lv);
  const float inv_l = out_scale / __uint_as_float(lv);
  // output half hh of the tile -> its 16 KB staging block, SW128 layout of the
  // out tensor map: row r at byte 128 r, 16-byte chunk k at k ^ (r % 8)
  uint8_t* stage = hh == 0 ? sm.q[t] : out_stage(sm, t);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t o[32];
    tmem_ld32(tmem + lanes32 + col_o(t) + 64 * hh + 32 * c, o);
    tmem_ld_wait(o);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int k = c * 4 + k4;
      *reinterpret_cast<uint4*>(stage + r * 128 + ((k ^ (r & 7)) << 4)) =
          make_uint4(w[4 * k4], w[4 * k4 + 1], w[4 * k4 + 2], w[4 * k4 + 3]);
    }
  }
  fence_proxy_async_smem();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(2 * BM) : "memory");
  if (wt == 0 && i == 0) {
    tma_store_4d(tm_o, smem_u32(sm.q[t]), 0, h, row0, b);  // rows >= N are clipped
    tma_store_4d(tm_o, smem_u32(out_stage(sm, t)), 64, h, row0, b);
    bulk_commit();
    bulk_wait_read_all();
  }
}

// tm_kr, tm_vr: the repair K and V tiles (REP; bf16 [B*H, R, 128], boxes of
// 64 dims x 128 rows); other instances never read them.
template <bool FP8, bool REP = false, bool SOL = false>
__global__ void __launch_bounds__((Roles<FP8, REP, SOL>::THREADS), 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr,
                const Params prm) {
  static_assert(FP8 || !REP, "the repair blocks belong to the FP8 kernel");
  static_assert(!FP8 || !SOL, "the block-sparse kernel is BF16");
  constexpr int KST = Traits<FP8>::KST, VST = Traits<FP8>::VST;
  using R = Roles<FP8, REP, SOL>;
  extern __shared__ uint8_t smem_raw[];
  Smem<FP8>& sm =
      *reinterpret_cast<Smem<FP8>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int b = bh / prm.H;
  const int h = bh - b * prm.H;
  const int q0 = blockIdx.x * CTA_ROWS;
  volatile int* ab = &sm.abort;

  if (threadIdx.x == 0) {
    for (int t = 0; t < TILES; ++t) {
      mbar_init(&sm.q_full[t], 1);
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], R::TILE_THREADS);
      mbar_init(&sm.o_full[t], 1);
    }
    for (int s = 0; s < KST; ++s) { mbar_init(&sm.k_full[s], 1); mbar_init(&sm.k_empty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_empty[s], 1); }
    for (int t = 0; t < TILES; ++t) {
      mbar_init(&sm.qbf_full[t], R::TILE_THREADS);
      mbar_init(&sm.s_free[t], R::TILE_THREADS);
      mbar_init(&sm.o_done[t], 1);
    }
    mbar_init(&sm.krep_full, 1);
    mbar_init(&sm.krep_empty, 1);
    mbar_init(&sm.vrep_full, 1);
    mbar_init(&sm.vrep_empty, 1);
    mbar_init(&sm.qbf_free, 1);
    for (int t = 0; t < TILES; ++t) mbar_init(&sm.lrep_full[t], R::TILE_THREADS);
    mbar_init(&sm.mma_drain, 1);
    mbar_init(&sm.mma_drain2, 1);
    mbar_init(&sm.never, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == R::LOAD_V && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_v);
    if (REP) tma_prefetch_desc(&tm_vr);
  }
  if (warp == R::LOAD_K && lane == 0) {
    tma_prefetch_desc(&tm_k);
    if (REP) tma_prefetch_desc(&tm_kr);
  }
  if (warp == R::MMA) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  // The grid is launched as a programmatic dependent of the kernel before it
  // in the stream (the prologue): the setup above overlaps that kernel's
  // tail, and no thread reads global memory before this wait.
  griddep_wait();
  // SOL: this CTA's list of key blocks; otherwise every block in order
  const uint16_t* lst = nullptr;
  int nkv = prm.nkv;
  if (SOL) {
    const size_t c = static_cast<size_t>(bh) * gridDim.x + blockIdx.x;
    lst = prm.sol_list + c * prm.sol_nb;
    nkv = __ldg(prm.sol_count + c);
  }

  if (prm.debug & 1) {  // FLUX_ATTN_DEBUG_FORCE_TIMEOUT: a wait nothing will satisfy
    if (threadIdx.x == 0) mbar_wait(&sm.never, 0, ab, prm.err);
    __syncthreads();
  }

  if (warp == R::LOAD_K) {
    if (lane == 0 && !*ab) load_k<FP8, REP, SOL>(sm, &tm_k, &tm_kr, bh, nkv, prm.nrep, lst, ab, prm.err);
    __syncwarp();
  } else if (warp == R::LOAD_V) {
    if (lane == 0 && !*ab)
      load_qv<FP8, REP, SOL>(sm, &tm_q, &tm_v, &tm_vr, q0, bh, b, h, nkv, prm.nrep, lst, ab, prm.err);
    __syncwarp();
  } else if (warp == R::MMA) {
    if constexpr (R::SPLIT) {
      if (!*ab) mma_split<REP, true>(sm, tmem, nkv, prm.nrep, ab, prm.err);  // the QKs (the whole warp: see mma_commit)
    } else {
      if (!*ab) mma_issuer(sm, tmem, nkv, ab, prm.err);  // the whole warp: see mma_commit
    }
    __syncwarp();
  } else if (R::SPLIT && warp == R::MMA_PV) {
    if constexpr (R::SPLIT) {
      if (!*ab) mma_split<REP, false>(sm, tmem, nkv, prm.nrep, ab, prm.err);  // the P.Vs and row sums
    }
    __syncwarp();
  } else if constexpr (R::SPLIT) {
    const int t = warp / (R::SOFTMAX_WARPS / TILES);  // query tile of this warp
    if (!*ab) softmax_epilogue_split<REP>(sm, tmem, prm, b, h, q0 + t * BM, t, nkv, ab, &tm_o);
  } else {
    const int t = warp >> 2;  // query tile of this warpgroup
    if (!*ab) softmax_epilogue<SOL>(sm, tmem, prm, b, h, q0 + t * BM, t, nkv, lst, ab, &tm_o);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == R::MMA) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace attn
}  // namespace flux
