// qkv_gemm.cuh -- QKV projection of the hidden states with the query/key
// normalisation and RoPE fused into the GEMM epilogue.
//
// "Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell
// GPUs", section "GEMM kernel optimisation": the QKV projection of a FLUX 3
// block is one GEMM whose epilogue applies the query/key normalisation and
// the rotary position embedding, so that attention reads finished Q and K.
//
//   y = x W^T (+ b)     x [M = B N, D] bf16, W [3 H 128, D] bf16 (a linear
//                       layer's [out, in] layout), b [3 H 128] fp32 or none
//   y = [Q | K | V], head h of each part owning features h*128 .. h*128+127
//   Q' = RoPE(RMSNorm(Q) w_q), K' = RoPE(RMSNorm(K) w_k)  -> bf16 [B, H, N, 128]
//   V                                                     -> bf16 [B, N, H, 128]
// (the layouts the attention kernel reads).
//
// Persistent kernel, one CTA per SM, tiles of 128 tokens x 256 output
// features (two heads), K in blocks of 64 (one 128-byte swizzle row of bf16):
//   warp 0     TMA producer: A (128 x 64) and B (256 x 64) per K block into a
//              4-stage ring (48 KB a stage)
//   warp 1     TMEM owner and MMA issuer (whole warp, one elected lane):
//              4 MMAs of 128 x 256 x 16 per K block into one of two TMEM
//              accumulators (2 x 256 columns), so that the epilogue of a tile
//              overlaps the MMAs of the next
//   warps 2-5  epilogue: thread r owns output row r (TMEM lane r); a 128-column
//              half of the accumulator is exactly one head, so the RMS is a
//              reduction inside one thread and the RoPE pairs are adjacent
//              columns of it; the (cos, sin) of a token come from a table
//              built per call (rope_table_kernel)
// Every wait is bounded and reports through the device error word.
#pragma once

#include "prologue.cuh"

namespace flux {
namespace qkv {

constexpr int BM = 128;                       // tokens per tile
constexpr int BN = 256;                       // output features per tile (two heads)
constexpr int BK = 64;                        // K per stage (128 bytes of bf16)
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;     // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;     // 32 KB
constexpr int THREADS = 192;
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_EPI0 = 2;
constexpr uint32_t TMEM_COLS = 512;           // two accumulators of 256 columns

struct __align__(1024) Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES], empty[STAGES];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

struct Params {
  const float* bias;        // [3 H 128] or nullptr
  const float* wq;          // [128]
  const float* wk;          // [128]
  const float2* rope;       // [N][64] (cos, sin) per token and pair
  __nv_bfloat16* qn;        // [B, H, N, 128]
  __nv_bfloat16* kn;        // [B, H, N, 128]
  __nv_bfloat16* v;         // [B, N, H, 128]
  uint32_t* err;
  uint32_t* amax;           // FP8: per-(b, h) |max| of the written Q', K', V, fp32 bits [B*H][3]
                            // (must be zero on entry); nullptr for BF16
  int M, N, H, D;           // tokens B*N, tokens per batch row, heads, hidden size
  int m_tiles, n_tiles;
  int group_m;              // token tiles per group of the tile order
  float eps;
};

// (cos, sin) of pair j of token n: pos_n[axis_j] * freq_j, precise sincosf
// (looked up in the handle's per-position table when the position is in it).
// Launched as one wave (a grid-stride loop over the N x 64 pairs, at most
// kTableBlocksPerSm blocks per SM), so that it may let the GEMM after it
// start early: the GEMM's producer and MMA warps do not read the table, and
// its epilogue waits for this grid (griddepcontrol.wait) before it does.
constexpr int kTableThreads = 256;
constexpr int kTableBlocksPerSm = 4;

__global__ void __launch_bounds__(kTableThreads)
    rope_table_kernel(TokenGeometry geo, int N, RopeTable tab, const float2* __restrict__ rot,
                      float2* __restrict__ out) {
  griddep_launch_dependents();
  const int total = N * (kHeadDim / 2);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int n = i / (kHeadDim / 2);
    const int j = i - n * (kHeadDim / 2);
    int p[3];
    token_position(geo, n, p);
    const int a = tab.axis[j];
    const int pos = a == 0 ? p[0] : (a == 1 ? p[1] : p[2]);
    if (rot != nullptr && static_cast<unsigned>(pos) < static_cast<unsigned>(kRotPositions)) {
      out[i] = __ldg(rot + pos * (kHeadDim / 2) + j);  // the same sincosf, tabulated per position
    } else {
      float s, c;
      sincosf(static_cast<float>(pos) * tab.freq[j], &s, &c);
      out[i] = make_float2(c, s);
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
}

// Tile order: groups of group_m token tiles; inside a group the token tile
// varies fastest, then the weight block.  When all of x fits in L2 next to
// the weights (4608 tokens: 28 MB) there is one group: every weight block is
// then shared by all token tiles in flight.  When it does not (16896 tokens:
// 104 MB), groups of 16 token tiles keep 12 MB of x resident while the group
// walks all weight blocks; one group over all of x would stream x through L2
// once per weight block.
constexpr int GROUP_M = 16;
constexpr size_t GROUP_X_BYTES = size_t(48) << 20;  // x rows that may form one group

__host__ __device__ inline int group_rows(int m_tiles, int d_model) {
  return static_cast<size_t>(m_tiles) * BM * d_model * 2 <= GROUP_X_BYTES ? m_tiles : GROUP_M;
}

__device__ __forceinline__ void tile_coords(const Params& p, int t, int& m0, int& n0) {
  const int per_group = p.group_m * p.n_tiles;
  const int g = t / per_group;
  const int rows = min(p.group_m, p.m_tiles - g * p.group_m);  // token tiles in this group
  const int local = t - g * per_group;
  m0 = (g * p.group_m + local % rows) * BM;
  n0 = (local / rows) * BN;
}

__device__ __forceinline__ void producer(Smem& sm, const CUtensorMap* ta, const CUtensorMap* tb, const Params& p,
                                         volatile int* ab) {
  const int nk = p.D / BK;
  const int tiles = p.m_tiles * p.n_tiles;
  int issued = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
    int m0, n0;
    tile_coords(p, t, m0, n0);
    for (int kb = 0; kb < nk; ++kb, ++issued) {
      const int s = issued % STAGES;
      const uint32_t u = issued / STAGES;
      if (u > 0 && !mbar_wait(&sm.empty[s], (u - 1) & 1, ab, p.err)) { ok = false; break; }
      mbar_arrive_expect_tx(&sm.full[s], A_BYTES + B_BYTES);
      tma_load_2d(smem_u32(sm.a[s]), ta, &sm.full[s], kb * BK, m0);
      tma_load_2d(smem_u32(sm.b[s]), tb, &sm.full[s], kb * BK, n0);
    }
  }
  for (int s = 0; s < STAGES; ++s) {  // nothing may still be landing when the CTA exits
    const int cnt = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
    if (cnt > 0) wait_drain(&sm.full[s], (cnt - 1) & 1, p.err);
  }
}

// Whole warp; one elected lane issues (see ptx.cuh).
__device__ __forceinline__ void mma_issuer(Smem& sm, uint32_t tmem, const Params& p, volatile int* ab) {
  constexpr uint32_t ID = idesc_f16(BM, BN, false);
  const int nk = p.D / BK;
  const int tiles = p.m_tiles * p.n_tiles;
  const uint64_t ad0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);
  const uint64_t bd0 = sdesc_sw128(smem_u32(sm.b[0]), 16, 1024);
  int consumed = 0;
  bool ok = true;
  for (int t = blockIdx.x, it = 0; t < tiles && ok; t += gridDim.x, ++it) {
    const int buf = it & 1;
    const uint32_t u = it >> 1;
    if (u > 0 && !mbar_wait(&sm.acc_empty[buf], (u - 1) & 1, ab, p.err)) break;
    tc_fence_after_sync();
    const uint32_t d = tmem + buf * BN;
    for (int kb = 0; kb < nk; ++kb, ++consumed) {
      const int s = consumed % STAGES;
      if (!mbar_wait(&sm.full[s], (consumed / STAGES) & 1, ab, p.err)) { ok = false; break; }
      tc_fence_after_sync();
      const uint64_t ad = ad0 + ((s * A_BYTES) >> 4);
      const uint64_t bd = bd0 + ((s * B_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_f16_ss(d, ad + ((kk * 32) >> 4), bd + ((kk * 32) >> 4), ID, (kb > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&sm.empty[s]);
    }
    if (ok) mma_commit(&sm.acc_full[buf]);
  }
  mma_commit(&sm.drain);
  wait_drain(&sm.drain, 0, p.err);
}

// |max| of the bf16 pairs in w, accumulated in m (two bf16 halves; non-negative
// bf16 values order like their bit patterns).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w) { return __vmaxu2(m, w & 0x7FFF7FFFu); }

// One head (128 columns) of row r: bias, then for Q and K the RMSNorm with
// its weight and the rotation, then bf16 stores of the 256-byte row.
// Returns the row's |max| of the values written (fp32 bits; 0 past the last
// row), for the FP8 path's per-head scales.
__device__ __forceinline__ uint32_t epilogue_head(const Params& p, uint32_t taddr, int col0, int m) {
  uint32_t y[128];
  tmem_ld128(taddr, y);
  tmem_ld_wait(y);
  const int F = p.H * kHeadDim;
  const int part = col0 / F;             // 0 Q, 1 K, 2 V
  const int h = (col0 - part * F) / kHeadDim;
  if (p.bias != nullptr) {
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + col0);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float4 bb = __ldg(b4 + i);
      y[4 * i] = __float_as_uint(__uint_as_float(y[4 * i]) + bb.x);
      y[4 * i + 1] = __float_as_uint(__uint_as_float(y[4 * i + 1]) + bb.y);
      y[4 * i + 2] = __float_as_uint(__uint_as_float(y[4 * i + 2]) + bb.z);
      y[4 * i + 3] = __float_as_uint(__uint_as_float(y[4 * i + 3]) + bb.w);
    }
  }
  if (m >= p.M) return 0u;
  const int b = m / p.N;
  const int n = m - b * p.N;
  uint32_t mx = 0u;
  if (part == 2) {
    uint4* dst = reinterpret_cast<uint4*>(p.v + ((static_cast<size_t>(b) * p.N + n) * p.H + h) * kHeadDim);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint4 u = make_uint4(pack_bf16x2(__uint_as_float(y[8 * i]), __uint_as_float(y[8 * i + 1])),
                                 pack_bf16x2(__uint_as_float(y[8 * i + 2]), __uint_as_float(y[8 * i + 3])),
                                 pack_bf16x2(__uint_as_float(y[8 * i + 4]), __uint_as_float(y[8 * i + 5])),
                                 pack_bf16x2(__uint_as_float(y[8 * i + 6]), __uint_as_float(y[8 * i + 7])));
      dst[i] = u;
      if (p.amax != nullptr)
        mx = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(mx, u.x), u.y), u.z), u.w);
    }
    return max(mx & 0xFFFFu, mx >> 16) << 16;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 128; ++i) ss = fmaf(__uint_as_float(y[i]), __uint_as_float(y[i]), ss);
  const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
  const float* w = part == 0 ? p.wq : p.wk;
  __nv_bfloat16* out = (part == 0 ? p.qn : p.kn) + ((static_cast<size_t>(b) * p.H + h) * p.N + n) * kHeadDim;
  const float4* cs4 = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(n) * (kHeadDim / 2));
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // 8 elements = 4 rotation pairs per step
    const float4 wa = __ldg(reinterpret_cast<const float4*>(w) + 2 * i);
    const float4 wb = __ldg(reinterpret_cast<const float4*>(w) + 2 * i + 1);
    const float4 c01 = __ldg(cs4 + 2 * i);      // (cos, sin) of pairs 4i, 4i+1
    const float4 c23 = __ldg(cs4 + 2 * i + 1);  // pairs 4i+2, 4i+3
    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    const float cv[4] = {c01.x, c01.z, c23.x, c23.z};
    const float sv[4] = {c01.y, c01.w, c23.y, c23.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y0 = __uint_as_float(y[8 * i + 2 * e]) * r * wv[2 * e];
      const float y1 = __uint_as_float(y[8 * i + 2 * e + 1]) * r * wv[2 * e + 1];
      o[e] = pack_bf16x2(y0 * cv[e] - y1 * sv[e], y0 * sv[e] + y1 * cv[e]);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    if (p.amax != nullptr)
      mx = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(mx, o[0]), o[1]), o[2]), o[3]);
  }
  return max(mx & 0xFFFFu, mx >> 16) << 16;
}

__device__ __forceinline__ void epilogue(Smem& sm, uint32_t tmem, const Params& p, volatile int* ab) {
  const int warp = threadIdx.x >> 5;
  const int q4 = warp & 3;                      // TMEM lane quarter this warp may access
  const int r = q4 * 32 + (threadIdx.x & 31);   // output row within the tile
  const int tiles = p.m_tiles * p.n_tiles;
  const int Nout = 3 * p.H * kHeadDim;
  for (int t = blockIdx.x, it = 0; t < tiles; t += gridDim.x, ++it) {
    const int buf = it & 1;
    const bool ok = mbar_wait(&sm.acc_full[buf], (it >> 1) & 1, ab, p.err);
    if (__any_sync(0xFFFFFFFFu, !ok)) break;
    tc_fence_after_sync();
    int m0, n0;
    tile_coords(p, t, m0, n0);
#pragma unroll 1
    for (int hs = 0; hs < BN / kHeadDim; ++hs) {
      const int col0 = n0 + hs * kHeadDim;
      if (col0 >= Nout) continue;  // tile-uniform
      const uint32_t am =
          epilogue_head(p, tmem + (static_cast<uint32_t>(q4 * 32) << 16) + buf * BN + hs * kHeadDim, col0, m0 + r);
      if (p.amax != nullptr) {
        // per-(b, h) amax: one atomic per warp when its 32 rows share a batch row
        const int F = p.H * kHeadDim;
        const int part = col0 / F, h = (col0 - part * F) / kHeadDim;
        const int b = min(m0 + r, p.M - 1) / p.N;
        const int b0 = __shfl_sync(0xFFFFFFFFu, b, 0);
        if (__all_sync(0xFFFFFFFFu, b == b0)) {
          uint32_t w = am;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) w = max(w, __shfl_xor_sync(0xFFFFFFFFu, w, off));
          if ((threadIdx.x & 31) == 0 && w != 0u) atomicMax(p.amax + (static_cast<size_t>(b0) * p.H + h) * 3 + part, w);
        } else if (am != 0u) {
          atomicMax(p.amax + (static_cast<size_t>(b) * p.H + h) * 3 + part, am);
        }
      }
    }
    tc_fence_before_sync();
    mbar_arrive(&sm.acc_empty[buf]);
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* ab = &sm.abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], BM);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  if (warp == WARP_TMA) {
    if (lane == 0) producer(sm, &tm_a, &tm_b, p, ab);
    __syncwarp();
  } else if (warp == WARP_MMA) {
    mma_issuer(sm, tmem, p, ab);
    __syncwarp();
  } else {
    griddep_wait();  // the (cos, sin) table comes from the kernel before this one
    epilogue(sm, tmem, p, ab);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace qkv
}  // namespace flux
