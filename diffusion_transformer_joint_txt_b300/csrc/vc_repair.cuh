// vc_repair.cuh -- VC-Attention FP8 repair: per (batch, head), the key
// tokens with the largest quantisation error attend with their exact K', V.
//
// "Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell
// GPUs", section "Quantized and sparse attention": VC-Attention FP8 takes a
// repair budget (vc_repair_budget, 0.005 in the page's configuration): up to
// that share of the tokens, the worst quantised ones, get their quantisation
// residual corrected.  Reading taken here (the page gives no formula): key
// token m of head (b, h) has the error
//     e_m = |k'_m - deq(k'_m)|^2 + |v_m - deq(v_m)|^2
// (written by the E4M3 quantisers as two arrays, errk and errv), the
// R = ceil(rho N) tokens with the largest e_m are repaired (equal errors: the
// lower token index first), and a repaired token takes part in the attention
// with its exact K' and V instead of their E4M3 codes; queries stay E4M3.
//
// Two kernels, one CTA per (b, h):
//   vc_select_kernel   the repair set, ascending, by a radix select on the
//                      fp32 error bits (non-negative floats order like their
//                      bits) and an ordered compaction that breaks ties by
//                      index: sel [B*H][R] int32
//   vc_repair_kernel   (1) moves the codes of the non-repaired tokens among
//                      the last R positions into the positions of the
//                      repaired tokens among the first N - R, so that the FP8
//                      keys of the attention are exactly the non-repaired
//                      ones, in [0, N - R) (attention is invariant under a
//                      permutation of its keys with their values);
//                      (2) writes the repaired rows in the units of the codes:
//                      krep = bf16(k' / s_k), vrep = bf16(v / s_v)
//                      [B*H][R][128], with k' recomputed exactly as the E4M3
//                      pass computes it (norm and rotation in fp32).
#pragma once

#include "quantize_fp8.cuh"

namespace flux {
namespace vc {

constexpr int kSelectThreads = 1024;
constexpr int kRepairThreads = 256;
constexpr int kMoveChunk = 1024;  // fillers noted per round of the repair kernel

// Exclusive prefix count of `flag` over the block's threads in thread order;
// *total receives the block's count.  Uses `warp_tot` (32 entries) of shared
// memory; every thread of the block must call it.
__device__ __forceinline__ uint32_t block_exclusive_count(bool flag, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, flag);
  const uint32_t in_warp = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(ballot);
  __syncthreads();
  uint32_t before = 0, all = 0;
  const int warps = blockDim.x >> 5;
  for (int w = 0; w < warps; ++w) {
    const uint32_t c = warp_tot[w];
    if (w < warp) before += c;
    all += c;
  }
  __syncthreads();  // warp_tot may be rewritten by the next call
  *total = all;
  return before + in_warp;
}

// Exclusive prefix sum of v over the block's threads in thread order (same
// rules as block_exclusive_count).
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  uint32_t before = 0, all = 0;
  const int warps = blockDim.x >> 5;
  for (int w = 0; w < warps; ++w) {
    const uint32_t c = warp_tot[w];
    if (w < warp) before += c;
    all += c;
  }
  __syncthreads();
  *total = all;
  return before + x - v;
}

// The selection's dynamic shared memory holds the error keys of up to this
// many tokens; longer sequences read them from global memory.
constexpr int kSelectSmemKeys = 48 * 1024;

// Repair set of head blockIdx.x: the R tokens of largest errk + errv,
// equal errors by lower index, written ascending to sel[blockIdx.x][0 .. R).
// 1 <= R <= N.  Dynamic shared memory: 4 N bytes when N <= kSelectSmemKeys
// (the keys, staged once), else none.
__global__ void __launch_bounds__(kSelectThreads)
    vc_select_kernel(const float* __restrict__ errk, const float* __restrict__ errv, int N, int R,
                     int32_t* __restrict__ sel) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_prefix, s_rank;
  const int lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(blockIdx.x) * N;
  const float* ek = errk + base;
  const float* ev = errv + base;
  const bool staged = N <= kSelectSmemKeys;
  if (staged)
    for (int m = threadIdx.x; m < N; m += blockDim.x) keys[m] = __float_as_uint(ek[m] + ev[m]);
  __syncthreads();
  auto key = [&](int m) { return staged ? keys[m] : __float_as_uint(ek[m] + ev[m]); };
  // Radix select, most significant byte first: the R-th largest key is
  // `prefix` once all four bytes are fixed; `rank` is its rank among the
  // keys that share the bytes fixed so far (1 = largest).  Errors of one head
  // share their top bytes, so the histogram adds are aggregated per warp.
  uint32_t prefix = 0, mask = 0, rank = static_cast<uint32_t>(R);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int m0 = 0; m0 < N; m0 += blockDim.x) {  // warp-uniform trip count
      const int m = m0 + threadIdx.x;
      const uint32_t u = m < N ? key(m) : 0u;
      const bool active = m < N && (u & mask) == prefix;
      const uint32_t am = __ballot_sync(0xFFFFFFFFu, active);
      if (active) {
        const uint32_t bin = (u >> shift) & 255u;
        const uint32_t peers = __match_any_sync(am, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t above = 0;
      int digit = 0;
      for (int dg = 255; dg >= 0; --dg) {
        if (above + hist[dg] >= rank) { digit = dg; break; }
        above += hist[dg];
      }
      s_prefix = prefix | (static_cast<uint32_t>(digit) << shift);
      s_rank = rank - above;
    }
    __syncthreads();
    prefix = s_prefix;
    rank = s_rank;
    mask |= 255u << shift;
  }
  // Every key above the threshold, and the first `rank` keys equal to it in
  // token order.  Thread t owns the contiguous tokens [t E, (t + 1) E): two
  // block scans give its first equal key's rank and its first output slot.
  const int E = (N + blockDim.x - 1) / blockDim.x;
  const int m0 = min(N, static_cast<int>(threadIdx.x) * E), m1 = min(N, m0 + E);
  uint32_t n_eq = 0;
  for (int m = m0; m < m1; ++m) n_eq += key(m) == prefix;
  uint32_t total;
  uint32_t eq_rank = block_exclusive_sum(n_eq, warp_tot, &total);
  uint32_t n_take = 0;
  for (int m = m0, r = eq_rank; m < m1; ++m) {
    const uint32_t u = key(m);
    n_take += u > prefix || (u == prefix && static_cast<uint32_t>(r) < rank);
    r += u == prefix;
  }
  uint32_t out = block_exclusive_sum(n_take, warp_tot, &total);
  for (int m = m0; m < m1; ++m) {
    const uint32_t u = key(m);
    const bool take = u > prefix || (u == prefix && eq_rank < rank);
    eq_rank += u == prefix;
    // exactly R keys are taken; the bound only keeps a wrong count in the row
    if (take && out < static_cast<uint32_t>(R)) sel[static_cast<size_t>(blockIdx.x) * R + out] = m;
    out += take;
  }
}

struct RepairArgs {
  const __nv_bfloat16* k;  // [B, N, H, 128]
  const __nv_bfloat16* v;  // [B, N, H, 128]
  const float* wk;         // [128]
  TokenGeometry geo;
  RopeTable tab;
  const float2* rot;       // rotation table (kRotPositions x 64), or nullptr
  int N, H, R;
  float eps;
  const float* scales;     // [B*H][3]
  const int32_t* sel;      // [B*H][R], ascending
  uint8_t* k8;             // [B*H][N][128]
  uint8_t* v8t;            // [B*H][128][npad]
  size_t npad;
  __nv_bfloat16* krep;     // [B*H][R][128]
  __nv_bfloat16* vrep;     // [B*H][R][128]
};

// First index i in sel[0 .. R) with sel[i] >= x.
__device__ __forceinline__ int lower_bound(const int32_t* sel, int R, int x) {
  int lo = 0, hi = R;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sel[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kRepairThreads) vc_repair_kernel(const RepairArgs a) {
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh - b * a.H;
  const int N = a.N, R = a.R, split = N - R;
  const int32_t* sel = a.sel + static_cast<size_t>(bh) * R;
  uint8_t* k8 = a.k8 + static_cast<size_t>(bh) * N * kHeadDim;
  uint8_t* v8t = a.v8t + static_cast<size_t>(bh) * kHeadDim * a.npad;
  // (1) The non-repaired tokens p among the last R positions fill, in order,
  // the positions of the repaired tokens among the first N - R.  Sources and
  // destinations are disjoint, so the moves do not race.  In chunks of
  // kMoveChunk fillers: each thread finds the fillers among its candidate
  // positions and notes (source, destination) at the filler's rank; then the
  // whole block moves them, a K row as 8 16-byte pieces and a V^T column as
  // 128 single bytes, one piece per thread and step.
  __shared__ int2 moves[kMoveChunk];
  const int low = lower_bound(sel, R, split);  // repaired tokens below N - R = fillers
  for (int c0 = 0; c0 < low; c0 += kMoveChunk) {
    const int cn = min(kMoveChunk, low - c0);
    for (int p = split + threadIdx.x; p < N; p += blockDim.x) {
      const int i = lower_bound(sel, R, p);       // repaired tokens below p
      if (i < R && sel[i] == p) continue;         // p is repaired itself
      const int r = (p - split) - (i - low);      // p's rank among the fillers: 0 <= r < low
      if (r < c0 || r >= c0 + cn) continue;
      const int dst = sel[r];
      moves[r - c0] = make_int2(p, dst >= 0 && dst < split ? dst : -1);
    }
    __syncthreads();
    constexpr int kPieces = kHeadDim / 16 + kHeadDim;  // K row pieces, then V^T bytes
    for (int w = threadIdx.x; w < cn * kPieces; w += blockDim.x) {
      const int f = w / kPieces, c = w - f * kPieces;
      const int2 mv = moves[f];
      if (mv.y < 0) continue;
      if (c < kHeadDim / 16) {
        reinterpret_cast<uint4*>(k8 + static_cast<size_t>(mv.y) * kHeadDim)[c] =
            reinterpret_cast<const uint4*>(k8 + static_cast<size_t>(mv.x) * kHeadDim)[c];
      } else {
        // V^T keeps the attention's key order within every 8 positions
        // (0 2 4 6 1 3 5 7; quantize_fp8.cuh): position p sits in column
        // 8 (p / 8) + 4 (p % 2) + (p % 8) / 2
        const size_t d = static_cast<size_t>(c - kHeadDim / 16) * a.npad;
        auto col = [](int p) { return 8 * (p >> 3) + 4 * (p & 1) + ((p & 7) >> 1); };
        v8t[d + col(mv.y)] = v8t[d + col(mv.x)];
      }
    }
    __syncthreads();
  }
  // (2) Repaired rows, a half-warp per row as in the E4M3 pass (lane l of the
  // half holds dims 8l .. 8l+7), two rows per warp step.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 15, half = lane >> 4;
  const int warps = blockDim.x >> 5;
  float w[8];
  {
    const float4* pw = reinterpret_cast<const float4*>(a.wk + sub * 8);
    const float4 w0 = __ldg(pw), w1 = __ldg(pw + 1);
    w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
    w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
  }
  const float inv_k = 1.f / __ldg(a.scales + 3 * bh + 1);
  const float inv_v = 1.f / __ldg(a.scales + 3 * bh + 2);
  for (int i0 = 2 * warp; i0 < R; i0 += 2 * warps) {  // warp-uniform
    const int i = i0 + half;
    const bool valid = i < R;
    const int n = min(max(sel[valid ? i : i0], 0), N - 1);
    const size_t src = ((static_cast<size_t>(b) * N + n) * a.H + h) * kHeadDim + sub * 8;
    float x[8], y[8];
    unpack8(*reinterpret_cast<const uint4*>(a.k + src), x);
    unpack8(*reinterpret_cast<const uint4*>(a.v + src), y);
    float cs[4], sn[4];
    lane_rotation(a.geo, a.tab, a.rot, n, sub, cs, sn);
    RotCoef kc;
    rot_coef(w, cs, sn, kc);
    norm_rope8_packed(x, kc, a.eps);  // all 32 lanes: the norm's shuffles
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[e] *= inv_k;
      y[e] *= inv_v;
    }
    if (valid) {
      const size_t dst = (static_cast<size_t>(bh) * R + i) * kHeadDim + sub * 8;
      *reinterpret_cast<uint4*>(a.krep + dst) = pack8(x);
      *reinterpret_cast<uint4*>(a.vrep + dst) = pack8(y);
    }
  }
}

}  // namespace vc
}  // namespace flux
