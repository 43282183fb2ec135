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
// K/V tile.  Warp roles:
//   warps 0-3  softmax + epilogue of query tile 0 (thread r owns row r, TMEM lane r;
//              the output tile leaves through shared memory and a TMA store)
//   warps 4-7  softmax + epilogue of query tile 1
//   warp 8     TMA producer of the K ring
//   warp 9     TMEM allocator and tcgen05.mma issuer (one elected lane)
//   warp 10    TMA producer of both Q tiles and of the V ring
// TMEM (512 columns): S_0 at 0, S_1 at 128, O_0 at 256, O_1 at 384.  The
// softmax of a tile overwrites its S with P, and the P.V MMA reads P straight
// from TMEM as its A operand.
//
// The MMA issue order is  QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) | ...
// so while the softmax of tile 0 works on S_0(j+1) the tensor core runs
// PV_1(j) and QK_1(j+1), and the other way round: each tile's softmax hides
// behind the other tile's two MMAs.  The MMAs of one
// thread complete in issue order, which is what makes two things safe:
// QK_t(j+1) overwrites the S_t columns that PV_t(j) reads P from, and the
// commit that signals S_t(j+1) also means that PV_t(j) has landed in O_t, so
// the softmax may rescale O_t as soon as it sees S_t(j+1).
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
// [B, H, 128, Npad] (kind::f8f6f4, K = 32 per MMA).  A 128 x 128 tile is one
// 16 KB SW128 block, K-major for all three (for V^T the keys are the K
// dimension of P.V).  P is E4M3 of 256 p, four per TMEM column; the row sum
// l adds the values the codes stand for, so that O = sum p~ v / sum p~ is a
// convex combination of the V rows whatever the rounding of P.  Scores are
// scaled by s_q s_k and the output by s_v (per-(b, h) scales).  The FP8
// softmax sums the P values in packed f16 (E4M3 values are exact in f16):
// decoding every code back to fp32 for the sum cost it a sixth of its
// throughput.
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
constexpr int WARP_LOAD_K = 4 * TILES;          // 8: TMA producer of the K ring
constexpr int WARP_MMA = WARP_LOAD_K + 1;       // 9: MMA issuer, TMEM owner
constexpr int WARP_LOAD_V = WARP_MMA + 1;       // 10: TMA producer of Q and the V ring
constexpr int THREADS = 32 * (WARP_LOAD_V + 1); // 352
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t HALF = BM * 128;  // one SW128 block: 128 rows x 128 bytes = 16 KB

__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }        // S_t / P_t
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; } // O_t

template <bool FP8>
struct Traits {
  static constexpr uint32_t TILE = FP8 ? HALF : 2 * HALF;  // bytes of one 128 x 128 operand tile
  static constexpr int KST = FP8 ? 4 : 3;                  // K ring stages
  static constexpr int VST = FP8 ? 4 : 2;                  // V ring stages
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
  uint64_t q_full[TILES];
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[TILES], p_full[TILES], o_full[TILES];
  uint64_t mma_drain;
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
  int N, H, nkv;
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

// K ring producer: K_j into stage j % KST once both tiles' QK of its
// previous occupant have completed.
template <bool FP8>
__device__ __forceinline__ void load_k(Smem<FP8>& sm, const CUtensorMap* tk, int bh, int nkv, volatile int* ab,
                                       uint32_t* err) {
  constexpr uint32_t TILE = Traits<FP8>::TILE;
  constexpr int KST = Traits<FP8>::KST;
  int issued = 0;
  for (int j = 0; j < nkv; ++j) {
    const int ks = j % KST;
    const uint32_t ku = j / KST;
    if (ku > 0 && !mbar_wait(&sm.k_empty[ks], (ku - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.k_full[ks], TILE);
    load_rows<FP8>(smem_u32(sm.k[ks]), tk, &sm.k_full[ks], j * BN, bh);
    ++issued;
  }
  drain_ring(sm.k_full, issued, err);
}

// Q and V ring producer: both Q tiles once, then V_j into stage j % VST once
// both tiles' PV of its previous occupant have completed.
template <bool FP8>
__device__ __forceinline__ void load_qv(Smem<FP8>& sm, const CUtensorMap* tq, const CUtensorMap* tv, int q0, int bh,
                                        int b, int h, int nkv, volatile int* ab, uint32_t* err) {
  constexpr uint32_t TILE = Traits<FP8>::TILE;
  constexpr int VST = Traits<FP8>::VST;
#pragma unroll
  for (int t = 0; t < TILES; ++t) {
    mbar_arrive_expect_tx(&sm.q_full[t], TILE);
    load_rows<FP8>(smem_u32(sm.q[t]), tq, &sm.q_full[t], q0 + t * BM, bh);
  }
  int issued = 0;
  for (int j = 0; j < nkv; ++j) {
    const int vs = j % VST;
    const uint32_t vu = j / VST;
    if (vu > 0 && !mbar_wait(&sm.v_empty[vs], (vu - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.v_full[vs], TILE);
    if (FP8) {
      // V^T [B*H, 128, Npad]: keys j*128.. are the inner (x) coordinate.
      tma_load_3d(smem_u32(sm.v[vs]), tv, &sm.v_full[vs], j * BN, 0, bh);
    } else {
      // V [B, N, H, 128] in place: box (64 dims, 1 head, 128 keys, 1 batch).
      tma_load_4d(smem_u32(sm.v[vs]), tv, &sm.v_full[vs], 0, h, j * BN, b);
      tma_load_4d(smem_u32(sm.v[vs]) + HALF, tv, &sm.v_full[vs], 64, h, j * BN, b);
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

// The MMA issuer: QK_0(0) QK_1(0), then PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1)
// for every j.  The whole warp runs this loop and one elected lane issues
// (ptx.cuh).  One thread issues for both tiles: the fixed order is what
// keeps the two tiles in turns (two independent issuers drift into step, and
// then both softmaxes run at once and compete for the same schedulers).
template <bool FP8>
__device__ __forceinline__ void mma_issuer(Smem<FP8>& sm, uint32_t tmem, int nkv, volatile int* ab,
                                           uint32_t* err) {
  constexpr uint32_t TILE = Traits<FP8>::TILE;
  constexpr int KST = Traits<FP8>::KST, VST = Traits<FP8>::VST;
  // Tile descriptors: K-major SW128 (SBO = 8 rows x 128 B) for Q, K and the
  // FP8 V^T; MN-major SW128 for the BF16 V (LBO = the other 64 head dims).
  uint64_t qd[TILES];
#pragma unroll
  for (int t = 0; t < TILES; ++t) qd[t] = sdesc_sw128(smem_u32(sm.q[t]), 16, 1024);
  const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
  const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), FP8 ? 16 : HALF, 1024);
  do {
    if (!mbar_wait(&sm.k_full[0], 0, ab, err)) break;
    bool ok = true;
#pragma unroll
    for (int t = 0; t < TILES && ok; ++t) {
      ok = mbar_wait(&sm.q_full[t], 0, ab, err);
      if (!ok) break;
      tc_fence_after_sync();
      issue_qk<FP8>(tmem + col_s(t), qd[t], kd0);
      mma_commit(&sm.s_full[t]);
    }
    if (!ok) break;
    mma_commit(&sm.k_empty[0]);
    for (int j = 0; j < nkv && ok; ++j) {
      const int vs = j % VST;
      if (!mbar_wait(&sm.v_full[vs], (j / VST) & 1, ab, err)) break;
      const uint64_t vd = desc_at(vd0, vs * TILE);
      const int jn = j + 1;
      const int ks = jn % KST;
      const uint64_t kd = desc_at(kd0, ks * TILE);
#pragma unroll
      for (int t = 0; t < TILES; ++t) {
        ok = mbar_wait(&sm.p_full[t], j & 1, ab, err);
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv<FP8>(tmem + col_o(t), tmem + col_s(t), vd, j > 0);
        if (t == TILES - 1) mma_commit(&sm.v_empty[vs]);
        if (jn < nkv) {
          if (t == 0) {
            ok = mbar_wait(&sm.k_full[ks], (jn / KST) & 1, ab, err);
            if (!ok) break;
            tc_fence_after_sync();
          }
          // In issue order after PV_t(j), which read P_t from these columns.
          issue_qk<FP8>(tmem + col_s(t), qd[t], kd);
          mma_commit(&sm.s_full[t]);
          if (t == TILES - 1) mma_commit(&sm.k_empty[ks]);
        } else {
          mma_commit(&sm.o_full[t]);
        }
      }
    }
  } while (0);
  // Drain every MMA this thread issued before TMEM is released.
  mma_commit(&sm.mma_drain);
  mbar_drain(&sm.mma_drain, 0, err);
}

// Two E4M3 codes (round to nearest even, saturating) of a float pair, a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// The values two E4M3 codes stand for, exact in f16.
__device__ __forceinline__ __half2 e4m3x2_value(uint32_t c) {
  return __half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c), __NV_E4M3));
}

// Softmax and epilogue of query tile `t` (128 threads, thread r = row r).
template <bool FP8>
__device__ __forceinline__ void softmax_epilogue(Smem<FP8>& sm, uint32_t tmem, const Params& prm, int b, int h,
                                                 int row0, int t, volatile int* ab, const CUtensorMap* tm_o) {
  const int r = threadIdx.x & (BM - 1);
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;  // TMEM lanes of this warp
  const uint32_t s_addr = tmem + lane_base + col_s(t);
  const uint32_t o_addr = tmem + lane_base + col_o(t);
  const int N = prm.N;
  const int nkv = prm.nkv;
  float sl2 = prm.scale_log2;
  float out_scale = 1.f;
  if (FP8) {
    const float* sc = prm.scales + 3 * (static_cast<size_t>(b) * prm.H + h);
    sl2 *= __ldg(sc) * __ldg(sc + 1);
    out_scale = __ldg(sc + 2);
  }
  // FP8 stores P as E4M3 of 256 p: the 2^8 factor is folded into the exponent
  // and cancels against l, which sums the same scaled values.
  constexpr float kPBias = FP8 ? 8.f : 0.f;
  constexpr float kRescale = Traits<FP8>::RESCALE;
  float m = -INFINITY;  // running max, in log2 units
  float l = 0.f;        // running row sum
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    ok = mbar_wait(&sm.s_full[t], j & 1, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) { ok = false; break; }
    tc_fence_after_sync();
    uint32_t s[BN];
    tmem_ld128(s_addr, s);
    tmem_ld_wait(s);
    const int valid = N - j * BN;  // keys of this tile that exist (> 0)
    if (valid < BN) {
#pragma unroll
      for (int i = 0; i < BN; ++i)
        if (i >= valid) s[i] = __float_as_uint(-INFINITY);
    }
    // Row max: four independent chains of three-input max (depth 16, not 127).
    float acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = fmaxf(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]));
#pragma unroll
    for (int i = 8; i < BN; i += 8) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        acc[c] = fmax3(acc[c], __uint_as_float(s[i + 2 * c]), __uint_as_float(s[i + 2 * c + 1]));
    }
    const float mx = fmax3(acc[0], acc[1], fmaxf(acc[2], acc[3]));
    const float m_tile = fmaxf(m, mx * sl2);
    // One decision per warp (TMEM moves are warp-wide); each row keeps its own alpha.
    const bool rescale = __any_sync(0xFFFFFFFFu, m_tile > m + kRescale);
    const float m_new = rescale ? m_tile : m;
    const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;  // 0 on the first tile
    const float nm = kPBias - m_new;
    // p = 2^(s sl2 - m): the argument of two scores per packed FMA; the row
    // sum in four packed accumulators.
    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float rs;
    if (FP8) {
      // P codes four per word (key 4i in the lowest byte); the row sum adds
      // the values of the codes, in eight packed f16 accumulators (each sums
      // at most 8 values <= 256: partial sums <= 2048, rounding <= 2^-11
      // relative per add) that are widened to fp32 once per block.
      uint32_t pk[32];
      __half2 hs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) hs[i] = __float2half2_rn(0.f);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x0, x1, x2, x3;
        fma2(x0, x1, __uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1]), sl2, sl2, nm, nm);
        fma2(x2, x3, __uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3]), sl2, sl2, nm, nm);
        const uint32_t lo = e4m3x2(ex2_approx(x0), ex2_approx(x1));
        const uint32_t hi = e4m3x2(ex2_approx(x2), ex2_approx(x3));
        pk[i] = lo | (hi << 16);
        hs[i & 7] = __hadd2(hs[i & 7], __hadd2(e4m3x2_value(lo), e4m3x2_value(hi)));
      }
      tmem_st32(s_addr, pk);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 f = __half22float2(hs[i]);
        sum[i] = f.x + f.y;
      }
    } else {
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
    rs = sum[0] + sum[1];
    l = l * alpha + rs;
    // O_t holds P_t(j-1) V(j-1) already (see the issue order), and nothing
    // else writes it until this thread arrives on p_full below.
    if (rescale && j > 0) {
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
  }
  if (ok) {
    ok = mbar_wait(&sm.o_full[t], 0, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
  }
  if (!ok) return;
  tc_fence_after_sync();
  const float inv_l = out_scale / l;
  // O tile (bf16, 32 KB) -> shared memory that no MMA or copy touches any
  // more, in the SW128 layout of the out tensor map: half c / 2 holds head
  // dims 64 (c / 2) .., row r at byte 128 r, its 16-byte chunk k at position
  // k ^ (r % 8).  BF16: the tile's own 32 KB Q buffer (its last QK completed
  // before the PV that signalled o_full).  FP8: a Q tile is only 16 KB, so
  // 32 KB of the K ring, idle once both tiles' last QK has completed (it
  // precedes PV_0(last) in issue order).  Then one thread writes the two
  // halves with TMA stores, which also clip rows >= N: whole 128-byte rows
  // instead of each thread's 16-byte pieces of rows H x 256 bytes apart.
  static_assert(!FP8 || Traits<FP8>::KST * Traits<FP8>::TILE >= TILES * 2 * HALF, "FP8 staging needs 64 KB of K ring");
  uint8_t* stage = FP8 ? &sm.k[0][0] + t * 2 * HALF : sm.q[t];
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
      *reinterpret_cast<uint4*>(stage + half * HALF + r * 128 + ((k ^ (r & 7)) << 4)) =
          make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
  fence_proxy_async_smem();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(BM) : "memory");
  if (r == 0) {
    tma_store_4d(tm_o, smem_u32(stage), 0, h, row0, b);          // rows >= N are clipped
    tma_store_4d(tm_o, smem_u32(stage) + HALF, 64, h, row0, b);
    bulk_commit();
    bulk_wait_all();
  }
}

template <bool FP8>
__global__ void __launch_bounds__(THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const Params prm) {
  constexpr int KST = Traits<FP8>::KST, VST = Traits<FP8>::VST;
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
      mbar_init(&sm.p_full[t], BM);
      mbar_init(&sm.o_full[t], 1);
    }
    for (int s = 0; s < KST; ++s) { mbar_init(&sm.k_full[s], 1); mbar_init(&sm.k_empty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_empty[s], 1); }
    mbar_init(&sm.mma_drain, 1);
    mbar_init(&sm.never, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == WARP_LOAD_V && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == WARP_LOAD_K && lane == 0) tma_prefetch_desc(&tm_k);
  if (warp == WARP_MMA) {
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

  if (prm.debug & 1) {  // FLUX_ATTN_DEBUG_FORCE_TIMEOUT: a wait nothing will satisfy
    if (threadIdx.x == 0) mbar_wait(&sm.never, 0, ab, prm.err);
    __syncthreads();
  }

  if (warp == WARP_LOAD_K) {
    if (lane == 0 && !*ab) load_k<FP8>(sm, &tm_k, bh, prm.nkv, ab, prm.err);
    __syncwarp();
  } else if (warp == WARP_LOAD_V) {
    if (lane == 0 && !*ab) load_qv<FP8>(sm, &tm_q, &tm_v, q0, bh, b, h, prm.nkv, ab, prm.err);
    __syncwarp();
  } else if (warp == WARP_MMA) {
    if (!*ab) mma_issuer<FP8>(sm, tmem, prm.nkv, ab, prm.err);  // the whole warp: see mma_commit
    __syncwarp();
  } else {
    const int t = warp >> 2;  // query tile of this warpgroup
    if (!*ab) softmax_epilogue<FP8>(sm, tmem, prm, b, h, q0 + t * BM, t, ab, &tm_o);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace attn
}  // namespace flux
