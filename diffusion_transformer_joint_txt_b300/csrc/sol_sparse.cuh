// sol_sparse.cuh -- Sol-Attention block mask: which 128-key blocks each
// 128-query block attends to.
//
// "Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell
// GPUs", section "Quantized and sparse attention": Sol-Attention (algorithm
// sol_attn, tau 1.0, disabled_until_timestep 0.96) skips blocks of the
// attention with a block-sparse kernel.  Reading taken here (the page gives no
// formula): per (b, h), queries and keys are cut into blocks of 128 tokens
// (the last one ragged); the pooled vector of a block is the mean of its
// normalised, rotated rows; query block i gives key block j the mass
//     mu_ij = c_j exp(q_bar_i . k_bar_j / sqrt(d)) / sum_j' c_j' exp(q_bar_i . k_bar_j' / sqrt(d))
// (c_j = keys in block j) and keeps the block when mu_ij >= tau / nb, plus
// always its block of largest mass (lowest index on ties).
//
// Three small kernels on the prologue's Q', K' (bf16 [B*H, N, 128]):
//   sol_pool_kernel   block means q_bar, k_bar, fp32 [B*H][nb][128]
//   sol_keep_kernel   keep [B*H][nb][nb] uint8 (1 = query block i keeps key block j)
//   sol_list_kernel   per attention CTA (query blocks 2c, 2c + 1) the union of
//                     the two rows' kept key blocks, ascending: entry = key
//                     block | keep-bit of query block 2c << 14 | of 2c + 1 << 15,
//                     list [B*H][ncta][nb] uint16, count [B*H][ncta] int32
#pragma once

#include "vc_repair.cuh"

namespace flux {
namespace sol {

constexpr int kBlock = 128;   // tokens per query / key block
constexpr int kThreads = 128;
constexpr int kMaxBlocks = 1 << 14;  // the list entry's 14-bit key block field
constexpr int kMaxNb = 2048;         // key blocks per head the keep kernel scores (262144 tokens)
constexpr int kPoolThreads = 256;

// Block means of Q' and K' of block blockIdx.x of head blockIdx.y: thread t
// sums the dim pair t % 64 (one bf16x2 word) over the rows t / 64, t / 64 + 4,
// ... (eight independent loads in flight), then the four row groups are
// added in a fixed order.
__global__ void __launch_bounds__(kPoolThreads)
    sol_pool_kernel(const __nv_bfloat16* __restrict__ qn, const __nv_bfloat16* __restrict__ kn, int N,
                    float* __restrict__ qbar, float* __restrict__ kbar) {
  __shared__ float2 part[2][kPoolThreads];
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
  const int dp = threadIdx.x & 63, rg = threadIdx.x >> 6;
  constexpr int kGroups = kPoolThreads / 64;
  const int r0 = blk * kBlock, r1 = min(N, r0 + kBlock);
  const size_t base = static_cast<size_t>(bh) * N * (kHeadDim / 2);  // in bf16x2 words
  const uint32_t* q = reinterpret_cast<const uint32_t*>(qn) + base;
  const uint32_t* k = reinterpret_cast<const uint32_t*>(kn) + base;
  float2 sq = make_float2(0.f, 0.f), sk = make_float2(0.f, 0.f);
#pragma unroll 8
  for (int r = r0 + rg; r < r1; r += kGroups) {
    const uint32_t a = __ldg(q + static_cast<size_t>(r) * (kHeadDim / 2) + dp);
    const uint32_t c = __ldg(k + static_cast<size_t>(r) * (kHeadDim / 2) + dp);
    sq.x += __uint_as_float(a << 16);
    sq.y += __uint_as_float(a & 0xFFFF0000u);
    sk.x += __uint_as_float(c << 16);
    sk.y += __uint_as_float(c & 0xFFFF0000u);
  }
  part[0][threadIdx.x] = sq;
  part[1][threadIdx.x] = sk;
  __syncthreads();
  if (rg == 0) {
    const float inv = 1.f / static_cast<float>(r1 - r0);
    for (int g = 1; g < kGroups; ++g) {
      const float2 a = part[0][g * 64 + dp], c = part[1][g * 64 + dp];
      sq.x += a.x; sq.y += a.y; sk.x += c.x; sk.y += c.y;
    }
    const size_t o = (static_cast<size_t>(bh) * nb + blk) * kHeadDim + 2 * dp;
    *reinterpret_cast<float2*>(qbar + o) = make_float2(sq.x * inv, sq.y * inv);
    *reinterpret_cast<float2*>(kbar + o) = make_float2(sk.x * inv, sk.y * inv);
  }
}

// Keep row of query block blockIdx.x of head blockIdx.y: each thread scores
// key blocks t, t + 128, ... once (into shared memory: at most kMaxNb), then
// block-wide max with its lowest index, the normaliser and the keep bytes.
__global__ void __launch_bounds__(kThreads)
    sol_keep_kernel(const float* __restrict__ qbar, const float* __restrict__ kbar, int N, float tau,
                    uint8_t* __restrict__ keep) {
  __shared__ float4 q4[kHeadDim / 4];
  __shared__ float sc[kMaxNb];
  __shared__ float red_v[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  const int i = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float4* kb = reinterpret_cast<const float4*>(kbar + static_cast<size_t>(bh) * nb * kHeadDim);
  if (tid < kHeadDim / 4)
    q4[tid] = reinterpret_cast<const float4*>(qbar + (static_cast<size_t>(bh) * nb + i) * kHeadDim)[tid];
  __syncthreads();
  const float scale = rsqrtf(static_cast<float>(kHeadDim));
  // scores in log units, with the log of the block's key count
  float mx = -INFINITY;
  int arg = 0x7FFFFFFF;
  for (int j = tid; j < nb; j += kThreads) {
    const float4* k = kb + static_cast<size_t>(j) * (kHeadDim / 4);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int e = 0; e < kHeadDim / 4; ++e) {
      const float4 a = q4[e], b = __ldg(k + e);
      s0 = fmaf(a.x, b.x, s0);
      s1 = fmaf(a.y, b.y, s1);
      s0 = fmaf(a.z, b.z, s0);
      s1 = fmaf(a.w, b.w, s1);
    }
    const int c = min(N, (j + 1) * kBlock) - j * kBlock;
    const float s = (s0 + s1) * scale + logf(static_cast<float>(c));
    sc[j] = s;
    if (s > mx) { mx = s; arg = j; }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float om = __shfl_xor_sync(0xFFFFFFFFu, mx, off);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, arg, off);
    if (om > mx || (om == mx && oi < arg)) { mx = om; arg = oi; }
  }
  if (lane == 0) { red_v[warp] = mx; red_i[warp] = arg; }
  __syncthreads();
  mx = red_v[0];
  arg = red_i[0];
  for (int w = 1; w < kThreads / 32; ++w)
    if (red_v[w] > mx || (red_v[w] == mx && red_i[w] < arg)) { mx = red_v[w]; arg = red_i[w]; }
  __syncthreads();
  float z = 0.f;
  for (int j = tid; j < nb; j += kThreads) z += expf(sc[j] - mx);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  if (lane == 0) red_v[warp] = z;
  __syncthreads();
  z = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) z += red_v[w];
  const float thr = tau / static_cast<float>(nb);
  uint8_t* row = keep + (static_cast<size_t>(bh) * nb + i) * nb;
  for (int j = tid; j < nb; j += kThreads) row[j] = (expf(sc[j] - mx) / z >= thr || j == arg) ? 1 : 0;
}

// Union list of the key blocks kept by query blocks 2c and 2c + 1 (c =
// blockIdx.x; the second may not exist) of head blockIdx.y, ascending.
__global__ void __launch_bounds__(kThreads)
    sol_list_kernel(const uint8_t* __restrict__ keep, int nb, uint16_t* __restrict__ list, int* __restrict__ count) {
  __shared__ uint32_t warp_tot[32];
  const int c = blockIdx.x, bh = blockIdx.y, ncta = gridDim.x;
  const uint8_t* r0 = keep + (static_cast<size_t>(bh) * nb + 2 * c) * nb;
  const bool has1 = 2 * c + 1 < nb;
  uint16_t* out = list + (static_cast<size_t>(bh) * ncta + c) * nb;
  uint32_t n = 0;
  for (int j0 = 0; j0 < nb; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    const uint32_t f = j < nb ? (r0[j] ? 1u : 0u) | ((has1 && r0[nb + j]) ? 2u : 0u) : 0u;
    uint32_t tot;
    const uint32_t pos = vc::block_exclusive_count(f != 0, warp_tot, &tot);
    if (f != 0) out[n + pos] = static_cast<uint16_t>(j | (f << 14));
    n += tot;
  }
  if (threadIdx.x == 0) count[static_cast<size_t>(bh) * ncta + c] = static_cast<int>(n);
}

}  // namespace sol
}  // namespace flux
