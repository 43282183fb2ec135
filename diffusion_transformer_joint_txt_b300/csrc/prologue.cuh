// prologue.cuh -- per-head Q/K RMSNorm followed by multi-axis RoPE.
//
// The QKV projection of a FLUX 3 Klein block carries query/key normalisation
// and rotary position embedding in its epilogue ("Speed up image generation
// with FLUX 3 Image Klein on NVIDIA Blackwell GPUs", section "GEMM kernel
// optimisation"); here it is a standalone memory-bound pass in front of the
// attention kernel.
//
//   in   q, k  bf16 [B, N, H, 128] (token-major, as a QKV projection writes them)
//   out  qn, kn bf16 [B, H, N, 128] (head-major, so that one attention tile is
//        one contiguous 32 KB block for TMA)
//
// A half-warp owns one head row: lane l of the half holds elements
// 8l .. 8l+7, i.e. the four adjacent pairs 4l .. 4l+3, which always fall
// inside one RoPE axis block (block edges 16 and 72 are multiples of 8).
// The rotation angles of a token do not depend on the head, so they are
// computed once per token and applied to all of its heads of Q and K.
#pragma once

#include "ptx.cuh"

namespace flux {

constexpr int kHeadDim = 128;

// Per rotation pair j (0..63): its frequency theta^(-2 jj / d_a) (jj = pair
// index inside axis block a) and the axis a whose position id it uses.
struct RopeTable {
  float freq[kHeadDim / 2];
  int axis[kHeadDim / 2];
};

// Where a token sits: explicit ids, or the [text | image | reference] geometry.
struct TokenGeometry {
  const int32_t* pos;   // [N, 3] or nullptr
  int txt, img_n, img_w, ref_w;
};

__device__ __forceinline__ void token_position(const TokenGeometry& g, int n, int p[3]) {
  if (g.pos != nullptr) {
    p[0] = __ldg(g.pos + 3 * n);
    p[1] = __ldg(g.pos + 3 * n + 1);
    p[2] = __ldg(g.pos + 3 * n + 2);
  } else if (n < g.txt) {
    p[0] = p[1] = p[2] = 0;
  } else if (n < g.txt + g.img_n) {
    const int t = n - g.txt;
    p[0] = 0;
    p[1] = t / g.img_w;
    p[2] = t % g.img_w;
  } else {
    const int t = n - g.txt - g.img_n;
    p[0] = 1;
    p[1] = t / g.ref_w;
    p[2] = t % g.ref_w;
  }
}

// Rotation angles of the four pairs a lane owns (pairs 4 sub .. 4 sub + 3);
// the axis of a pair picks its position id with selects, not an indexed
// local array.
__device__ __forceinline__ void lane_rotation(const TokenGeometry& geo, const RopeTable& tab, int n, int sub,
                                              float (&c)[4], float (&s)[4]) {
  int p[3];
  token_position(geo, n, p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = sub * 4 + i;
    const int a = tab.axis[j];
    const int pos = a == 0 ? p[0] : (a == 1 ? p[1] : p[2]);
    sincosf(static_cast<float>(pos) * tab.freq[j], &s[i], &c[i]);
  }
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// RMSNorm over the 128 elements held by a half-warp, weight, then rotation.
__device__ __forceinline__ void norm_rope8(float (&x)[8], const float (&w)[8], const float (&c)[4],
                                           const float (&s)[4], float eps) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float r = rsqrtf(ss * (1.0f / kHeadDim) + eps);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float y0 = x[2 * i] * r * w[2 * i];
    const float y1 = x[2 * i + 1] * r * w[2 * i + 1];
    x[2 * i] = y0 * c[i] - y1 * s[i];
    x[2 * i + 1] = y0 * s[i] + y1 * c[i];
  }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

// Streaming layout: a persistent block per SM.  One producer warp copies
// chunks of T consecutive tokens of q and of k -- T x H x 256 contiguous bytes
// each, since a token's heads are adjacent in [B, N, H, 128] -- into a
// two-stage shared-memory ring with single bulk copies.  The sixteen compute
// warps split a chunk token by token: 16 / T warps per token, each taking
// every (16 / T)-th head pair of it, so that a warp computes its token's
// (cos, sin) pairs and (b, n) once per chunk and then only normalises,
// rotates and stores rows (a half-warp per head row, read from shared memory,
// written head-major).  The copies of the next chunk are in flight while a
// chunk is computed.
constexpr int kProWarps = 16;                        // compute warps
constexpr int kProTokens = 8;                        // tokens per chunk at most
constexpr int kPrologueThreads = 32 * (kProWarps + 1);
constexpr int kProStages = 2;
constexpr int kProStageBytes = 96 * 1024;            // q + k rows of one chunk
constexpr int kProMaxHeads = kProStageBytes / (2 * kHeadDim * 2);  // 192: one token per chunk

// Tokens per chunk for H heads (>= 1 for H <= kProMaxHeads).
__host__ __device__ constexpr int prologue_chunk_tokens(int H) {
  return kProStageBytes / (2 * kHeadDim * 2 * H) < kProTokens ? kProStageBytes / (2 * kHeadDim * 2 * H)
                                                               : kProTokens;
}

__global__ void __launch_bounds__(kPrologueThreads, 1)
    qk_norm_rope_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                        const float* __restrict__ wq, const float* __restrict__ wk, TokenGeometry geo,
                        int B, int N, int H, float eps, RopeTable tab, __nv_bfloat16* __restrict__ qn,
                        __nv_bfloat16* __restrict__ kn, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t ring[];  // stage s: [T][H][128] q rows, then the same for k
  __shared__ uint64_t full[kProStages], empty[kProStages];
  __shared__ int abort_flag;
  const int T = prologue_chunk_tokens(H);
  const long long tokens = static_cast<long long>(B) * N;
  const int nchunks = static_cast<int>((tokens + T - 1) / T);
  const uint32_t part = static_cast<uint32_t>(T) * H * kHeadDim * 2;  // bytes of q (or k) rows per stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* ab = &abort_flag;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kProStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kProWarps);
    }
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == kProWarps) {  // producer
    if (lane == 0) {
      int issued = 0;
      for (int c = blockIdx.x, i = 0; c < nchunks; c += gridDim.x, ++i) {
        const int s = i % kProStages;
        const uint32_t u = i / kProStages;
        if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1, ab, err)) break;
        const long long t0 = static_cast<long long>(c) * T;
        const uint32_t bytes = static_cast<uint32_t>(min(static_cast<long long>(T), tokens - t0)) * H * kHeadDim * 2;
        const size_t off = static_cast<size_t>(t0) * H * kHeadDim;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        bulk_load(smem_u32(ring + s * 2 * part), q + off, bytes, &full[s]);
        bulk_load(smem_u32(ring + s * 2 * part + part), k + off, bytes, &full[s]);
        ++issued;
      }
      for (int s = 0; s < kProStages; ++s) {  // no copy may still be writing when the block exits
        const int cnt = issued > s ? (issued - s + kProStages - 1) / kProStages : 0;
        if (cnt > 0) {
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, (cnt - 1) & 1))
            if (globaltimer_ns() - t0 > kWaitLimitNs) { atomicOr(err, kErrTimeout); break; }
        }
      }
    }
    return;
  }

  const int sub = lane & 15;
  const int half = lane >> 4;
  const int G = kProWarps / T;   // warps per token
  const int tl = warp / G;       // this warp's token within each chunk (idle when >= T)
  const int g = warp - tl * G;   // first head pair of this warp; step G
  float w_q[8], w_k[8];
  {
    const float4* a = reinterpret_cast<const float4*>(wq + sub * 8);
    const float4* bb = reinterpret_cast<const float4*>(wk + sub * 8);
    const float4 a0 = __ldg(a), a1 = __ldg(a + 1), b0 = __ldg(bb), b1 = __ldg(bb + 1);
    w_q[0] = a0.x; w_q[1] = a0.y; w_q[2] = a0.z; w_q[3] = a0.w;
    w_q[4] = a1.x; w_q[5] = a1.y; w_q[6] = a1.z; w_q[7] = a1.w;
    w_k[0] = b0.x; w_k[1] = b0.y; w_k[2] = b0.z; w_k[3] = b0.w;
    w_k[4] = b1.x; w_k[5] = b1.y; w_k[6] = b1.z; w_k[7] = b1.w;
  }
  const size_t head_stride = static_cast<size_t>(N) * kHeadDim;  // elements between heads of Q' / K'
  for (int c = blockIdx.x, i = 0; c < nchunks; c += gridDim.x, ++i) {
    const int s = i % kProStages;
    const bool ok = mbar_wait(&full[s], (i / kProStages) & 1, ab, err);
    if (__any_sync(0xFFFFFFFFu, !ok)) break;
    const long long token = static_cast<long long>(c) * T + tl;
    if (tl < T && token < tokens) {
      const int b = static_cast<int>(token / N);
      const int n = static_cast<int>(token - static_cast<long long>(b) * N);
      float cs[4], sn[4];
      lane_rotation(geo, tab, n, sub, cs, sn);
      const uint8_t* sq = ring + s * 2 * part + (static_cast<size_t>(tl) * H * kHeadDim + sub * 8) * 2;
      __nv_bfloat16* oq = qn + (static_cast<size_t>(b) * H * N + n) * kHeadDim + sub * 8;
      __nv_bfloat16* ok_ = kn + (static_cast<size_t>(b) * H * N + n) * kHeadDim + sub * 8;
      // The whole warp works on one head pair at a time (norm_rope8 shuffles
      // across it); a half-warp past the last head computes on zeros and
      // stores nothing.
      // two head pairs per step: four independent rows, so that their
      // shuffle reductions overlap
      for (int hp = 2 * g; hp < H; hp += 4 * G) {
        const int h0 = hp + half, h1 = hp + 2 * G + half;
        uint4 uq0 = make_uint4(0, 0, 0, 0), uk0 = uq0, uq1 = uq0, uk1 = uq0;
        if (h0 < H) {
          uq0 = *reinterpret_cast<const uint4*>(sq + h0 * kHeadDim * 2);
          uk0 = *reinterpret_cast<const uint4*>(sq + part + h0 * kHeadDim * 2);
        }
        if (h1 < H) {
          uq1 = *reinterpret_cast<const uint4*>(sq + h1 * kHeadDim * 2);
          uk1 = *reinterpret_cast<const uint4*>(sq + part + h1 * kHeadDim * 2);
        }
        float xq0[8], xk0[8], xq1[8], xk1[8];
        unpack8(uq0, xq0);
        unpack8(uk0, xk0);
        unpack8(uq1, xq1);
        unpack8(uk1, xk1);
        norm_rope8(xq0, w_q, cs, sn, eps);
        norm_rope8(xk0, w_k, cs, sn, eps);
        norm_rope8(xq1, w_q, cs, sn, eps);
        norm_rope8(xk1, w_k, cs, sn, eps);
        if (h0 < H) {
          *reinterpret_cast<uint4*>(oq + h0 * head_stride) = pack8(xq0);
          *reinterpret_cast<uint4*>(ok_ + h0 * head_stride) = pack8(xk0);
        }
        if (h1 < H) {
          *reinterpret_cast<uint4*>(oq + h1 * head_stride) = pack8(xq1);
          *reinterpret_cast<uint4*>(ok_ + h1 * head_stride) = pack8(xk1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

}  // namespace flux
