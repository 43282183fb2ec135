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
// One warp per token (b, n).  The rotation angles of a token do not depend on
// the head, so each warp computes its 64 (cos, sin) pairs once and applies
// them to all H heads of Q and K.  A half-warp owns one head row: lane l of
// the half holds elements 8l .. 8l+7, i.e. the four adjacent pairs 4l .. 4l+3,
// which always fall inside one RoPE axis block (block edges 16 and 72 are
// multiples of 8).
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

constexpr int kPrologueThreads = 256;

__global__ void __launch_bounds__(kPrologueThreads)
    qk_norm_rope_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                        const float* __restrict__ wq, const float* __restrict__ wk, TokenGeometry geo,
                        int B, int N, int H, float eps, RopeTable tab, __nv_bfloat16* __restrict__ qn,
                        __nv_bfloat16* __restrict__ kn) {
  const int token = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  if (token >= B * N) return;  // warp-uniform
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const int half = lane >> 4;
  const int b = token / N;
  const int n = token - b * N;

  int p[3];
  token_position(geo, n, p);
  float c[4], s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = sub * 4 + i;
    const float ang = static_cast<float>(p[tab.axis[j]]) * tab.freq[j];
    sincosf(ang, &s[i], &c[i]);
  }
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

  const size_t in_row0 = (static_cast<size_t>(b) * N + n) * H;
#pragma unroll 2
  for (int hp = 0; hp < H; hp += 2) {
    const int h = hp + half;
    const bool valid = h < H;
    uint4 uq = make_uint4(0, 0, 0, 0), uk = make_uint4(0, 0, 0, 0);
    const size_t src = (in_row0 + h) * kHeadDim + sub * 8;
    if (valid) {
      uq = __ldg(reinterpret_cast<const uint4*>(q + src));
      uk = __ldg(reinterpret_cast<const uint4*>(k + src));
    }
    float xq[8], xk[8];
    unpack8(uq, xq);
    unpack8(uk, xk);
    norm_rope8(xq, w_q, c, s, eps);
    norm_rope8(xk, w_k, c, s, eps);
    if (valid) {
      const size_t dst = ((static_cast<size_t>(b) * H + h) * N + n) * kHeadDim + sub * 8;
      *reinterpret_cast<uint4*>(qn + dst) = pack8(xq);
      *reinterpret_cast<uint4*>(kn + dst) = pack8(xk);
    }
  }
}

}  // namespace flux
