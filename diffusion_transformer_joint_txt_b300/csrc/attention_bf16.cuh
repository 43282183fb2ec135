// attention_bf16.cuh -- joint (non-causal) flash attention on sm_103a tensor cores.
//
// Joint attention of "Speed up image generation with FLUX 3 Image Klein on
// NVIDIA Blackwell GPUs" (section "FLUX 3 inference with TensorRT LLM
// VisualGen"): every query token of [text | image | reference] attends to
// every key token of the same (batch, head); no mask.  The page measures the
// BF16 "VANILLA" attention at about 60 % of DiT kernel time (section
// "Quantized and sparse attention"); this kernel is that BF16 step.
//
// One CTA = one 128-row query tile of one (b, h).  Warp roles:
//   warps 0-3  softmax + epilogue, thread t owns query row t (TMEM lane t)
//   warp 4     TMA producer: Q once, then K_j / V_j into 2-stage rings
//   warp 5     TMEM allocator and single-thread tcgen05.mma issuer
// TMEM (512 columns): S_0 at 0, S_1 at 128 (S_j double-buffered so that
// S_{j+1} = Q K_{j+1}^T runs while the softmax works on S_j), O at 256.
// The softmax overwrites S_j with P_j (bf16, two per 32-bit column) and the
// P.V MMA reads its A operand straight from TMEM.
//
// Shared-memory layout of a 128 x 128 bf16 tile: two 16 KB halves (head-dim
// columns 0-63, 64-127), each 128 rows x 128 bytes with the 128-byte TMA
// swizzle, which is the canonical SW128 layout the MMA descriptors describe
// (K-major for Q and K; MN-major for V, whose head dim is the N of P.V).
//
// Every wait is bounded (ptx.cuh); a wait that runs out sets the CTA abort
// flag and the error word, all roles stop issuing, drain what they issued,
// free TMEM and return.
#pragma once

#include "ptx.cuh"

namespace flux {
namespace attn {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int HD = 128;  // head dim
constexpr int KST = 2;   // K ring stages
constexpr int VST = 2;   // V ring stages
constexpr uint32_t TILE = BM * HD * 2;  // 32 KB
constexpr uint32_t HALF = TILE / 2;     // one 64-column swizzle block: 128 rows x 128 B
constexpr int THREADS = 192;
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;

struct __align__(1024) Smem {
  uint8_t q[TILE];
  uint8_t k[KST][TILE];
  uint8_t v[VST][TILE];
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint64_t mma_drain;
  uint64_t never;  // nothing arrives here (forced-timeout debug path)
  uint32_t tmem_base;
  int abort;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + slack to align the base to 1024

struct Params {
  __nv_bfloat16* out;  // [B, N, H, 128]
  uint32_t* err;
  int N, H, nkv;
  float scale_log2;    // log2(e) / sqrt(128)
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

__device__ __forceinline__ void producer(Smem& sm, const CUtensorMap* tq, const CUtensorMap* tk,
                                         const CUtensorMap* tv, int q0, int bh, int b, int h, int nkv,
                                         volatile int* ab, uint32_t* err) {
  mbar_arrive_expect_tx(&sm.q_full, TILE);
  tma_load_3d(smem_u32(sm.q), tq, &sm.q_full, 0, q0, bh);
  tma_load_3d(smem_u32(sm.q) + HALF, tq, &sm.q_full, 64, q0, bh);
  int k_issued = 0, v_issued = 0;
  for (int j = 0; j < nkv; ++j) {
    const int ks = j % KST;
    const uint32_t ku = j / KST;
    if (ku > 0 && !mbar_wait(&sm.k_empty[ks], (ku - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.k_full[ks], TILE);
    tma_load_3d(smem_u32(sm.k[ks]), tk, &sm.k_full[ks], 0, j * BN, bh);
    tma_load_3d(smem_u32(sm.k[ks]) + HALF, tk, &sm.k_full[ks], 64, j * BN, bh);
    ++k_issued;
    const int vs = j % VST;
    const uint32_t vu = j / VST;
    if (vu > 0 && !mbar_wait(&sm.v_empty[vs], (vu - 1) & 1, ab, err)) break;
    mbar_arrive_expect_tx(&sm.v_full[vs], TILE);
    tma_load_4d(smem_u32(sm.v[vs]), tv, &sm.v_full[vs], 0, h, j * BN, b);
    tma_load_4d(smem_u32(sm.v[vs]) + HALF, tv, &sm.v_full[vs], 64, h, j * BN, b);
    ++v_issued;
  }
  // Drain: the latest phase of every barrier a copy was issued on has completed.
  mbar_drain(&sm.q_full, 0, err);
  for (int s = 0; s < KST; ++s) {
    const int cnt = k_issued > s ? (k_issued - s + KST - 1) / KST : 0;
    if (cnt > 0) mbar_drain(&sm.k_full[s], (cnt - 1) & 1, err);
  }
  for (int s = 0; s < VST; ++s) {
    const int cnt = v_issued > s ? (v_issued - s + VST - 1) / VST : 0;
    if (cnt > 0) mbar_drain(&sm.v_full[s], (cnt - 1) & 1, err);
  }
}

// S = Q K^T: 8 MMAs of 128 x 128 x 16.  Step kk covers head dims 16kk..16kk+15:
// half kk/4 of the tile, 32-byte offset (kk%4) inside the 128-byte swizzle row.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t qa, uint32_t ka) {
  constexpr uint32_t ID = idesc_f16(BM, BN, false);
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
    mma_f16_ss(d_tmem, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), ID, kk > 0);
  }
}

// O (+)= P V: 8 MMAs of 128 x 128 x 16.  Step kk covers keys 16kk..16kk+15:
// P columns 8kk.. (two bf16 per column), V rows 16kk.. (16 rows x 128 B = 2 KB);
// V is MN-major: LBO = next 64 head-dim columns (the other half), SBO = next 8 keys.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t va, bool accumulate) {
  constexpr uint32_t ID = idesc_f16(BM, HD, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_f16_ts(o_tmem, p_tmem + kk * 8, sdesc_sw128(va + kk * 2048, HALF, 1024), ID,
               (accumulate || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ void mma_issuer(Smem& sm, uint32_t tmem, int nkv, volatile int* ab, uint32_t* err) {
  const uint32_t qa = smem_u32(sm.q);
  do {
    if (!mbar_wait(&sm.q_full, 0, ab, err)) break;
    if (!mbar_wait(&sm.k_full[0], 0, ab, err)) break;
    tc_fence_after_sync();
    issue_qk(tmem + COL_S0, qa, smem_u32(sm.k[0]));
    mma_commit(&sm.s_full[0]);
    mma_commit(&sm.k_empty[0]);
    for (int j = 0; j < nkv; ++j) {
      if (j + 1 < nkv) {
        const int jn = j + 1;
        const int ks = jn % KST;
        if (!mbar_wait(&sm.k_full[ks], (jn / KST) & 1, ab, err)) break;
        tc_fence_after_sync();
        // S buffer jn&1 last held P_{j-1}, whose P.V MMA was issued before this one.
        issue_qk(tmem + ((jn & 1) ? COL_S1 : COL_S0), qa, smem_u32(sm.k[ks]));
        mma_commit(&sm.s_full[jn & 1]);
        mma_commit(&sm.k_empty[ks]);
      }
      if (!mbar_wait(&sm.p_full[j & 1], (j >> 1) & 1, ab, err)) break;
      const int vs = j % VST;
      if (!mbar_wait(&sm.v_full[vs], (j / VST) & 1, ab, err)) break;
      tc_fence_after_sync();
      issue_pv(tmem + COL_O, tmem + ((j & 1) ? COL_S1 : COL_S0), smem_u32(sm.v[vs]), j > 0);
      mma_commit(&sm.o_done);
      mma_commit(&sm.v_empty[vs]);
    }
  } while (0);
  // Drain every MMA this thread issued before TMEM is released.
  mma_commit(&sm.mma_drain);
  mbar_drain(&sm.mma_drain, 0, err);
}

__device__ __forceinline__ void softmax_epilogue(Smem& sm, uint32_t tmem, const Params& prm, int b, int h,
                                                 int q0, volatile int* ab) {
  const int t = threadIdx.x;  // 0..127
  const int warp = t >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int N = prm.N;
  const int nkv = prm.nkv;
  const float sl2 = prm.scale_log2;
  float m = -INFINITY;  // running max, in log2 units
  float l = 0.f;        // running row sum
  bool ok = true;
  for (int j = 0; j < nkv && ok; ++j) {
    const uint32_t scol = (j & 1) ? COL_S1 : COL_S0;
    ok = mbar_wait(&sm.s_full[j & 1], (j >> 1) & 1, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) { ok = false; break; }
    tc_fence_after_sync();
    float s[BN];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + scol + c * 32, r);
      tmem_ld_wait(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
    }
    const int valid = N - j * BN;  // keys of this tile that exist (> 0)
    if (valid < BN) {
#pragma unroll
      for (int i = 0; i < BN; ++i)
        if (i >= valid) s[i] = -INFINITY;
    }
    float mx = s[0];
#pragma unroll
    for (int i = 1; i < BN; ++i) mx = fmaxf(mx, s[i]);
    const float m_new = fmaxf(m, mx * sl2);
    const float alpha = ex2_approx(m - m_new);  // 0 on the first tile
    float rs = 0.f;
    uint32_t pk[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) {
      const float p0 = ex2_approx(fmaf(s[2 * i], sl2, -m_new));
      const float p1 = ex2_approx(fmaf(s[2 * i + 1], sl2, -m_new));
      rs += p0 + p1;
      pk[i] = pack_bf16x2(p0, p1);
    }
    l = l * alpha + rs;
    {
      uint32_t r0[32], r1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) { r0[i] = pk[i]; r1[i] = pk[32 + i]; }
      tmem_st32(tmem + lane_base + scol, r0);
      tmem_st32(tmem + lane_base + scol + 32, r1);
      tmem_st_wait();
    }
    // Every phase of o_done is confirmed in order (a parity wait is only exact
    // when the barrier is at most one phase away), then O is rescaled where
    // the running max moved.  P.V of tile j-1 has landed at this point.
    if (j > 0) {
      ok = mbar_wait(&sm.o_done, (j - 1) & 1, ab, prm.err);
      if (__any_sync(0xFFFFFFFFu, !ok)) { ok = false; break; }
      tc_fence_after_sync();
      if (__any_sync(0xFFFFFFFFu, m_new > m)) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + COL_O + c * 32, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + lane_base + COL_O + c * 32, r);
        }
        tmem_st_wait();
      }
    }
    m = m_new;
    tc_fence_before_sync();
    mbar_arrive(&sm.p_full[j & 1]);
  }
  if (ok) {
    ok = mbar_wait(&sm.o_done, (nkv - 1) & 1, ab, prm.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) ok = false;
  }
  if (!ok) return;
  tc_fence_after_sync();
  const float inv_l = 1.f / l;
  const int row = q0 + t;
  __nv_bfloat16* dst = prm.out + ((static_cast<size_t>(b) * N + row) * prm.H + h) * HD;
#pragma unroll
  for (int c = 0; c < HD / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tmem + lane_base + COL_O + c * 32, r);
    tmem_ld_wait(r);
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      o[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
    if (row < N) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int b = bh / prm.H;
  const int h = bh - b * prm.H;
  const int q0 = blockIdx.x * BM;
  volatile int* ab = &sm.abort;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < KST; ++s) { mbar_init(&sm.k_full[s], 1); mbar_init(&sm.k_empty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&sm.s_full[s], 1); mbar_init(&sm.p_full[s], BM); }
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.mma_drain, 1);
    mbar_init(&sm.never, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (prm.debug & 1) {  // FLUX_ATTN_DEBUG_FORCE_TIMEOUT: a wait nothing will satisfy
    if (threadIdx.x == 0) mbar_wait(&sm.never, 0, ab, prm.err);
    __syncthreads();
  }

  if (warp == WARP_TMA) {
    if (lane == 0 && !*ab) producer(sm, &tm_q, &tm_k, &tm_v, q0, bh, b, h, prm.nkv, ab, prm.err);
    __syncwarp();
  } else if (warp == WARP_MMA) {
    if (lane == 0 && !*ab) mma_issuer(sm, tmem, prm.nkv, ab, prm.err);
    __syncwarp();
  } else {
    if (!*ab) softmax_epilogue(sm, tmem, prm, b, h, q0, ab);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace attn
}  // namespace flux
