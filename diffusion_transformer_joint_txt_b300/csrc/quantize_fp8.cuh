// quantize_fp8.cuh -- FP8 (E4M3) prologue: per-(batch, head) amax of the
// normalised, rotated Q', K' and of V, then E4M3 codes of x / scale with
// scale = amax / 448 (1 when amax == 0).
//
// "Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell
// GPUs", section "Quantized and sparse attention": the FP8 attention runs Q.K
// and P.V with FP8 Q, K and V (qk_dtype fp8, v_dtype fp8); the quantisation
// comes after the query/key normalisation and RoPE of section "GEMM kernel
// optimisation".  Scales are per (batch, head) and per tensor.
//
// Two passes over q, k, v (bf16 [B, N, H, 128]):
//   fp8_amax_kernel   recomputes Q', K' in fp32 (the same norm + rotation as
//                     qk_norm_rope_kernel) and reduces |Q'|, |K'|, |V| per
//                     (b, h) into amax[B*H][3] (fp32 bit patterns; positive
//                     floats order like their bits, so atomicMax on the
//                     bits is a float max).  amax must be zero on entry.
//   fp8_quant_kernel  recomputes Q', K', scales and writes
//                       q8, k8   E4M3 [B, H, N, 128]
//                       scales   fp32 [B, H, 3] = (s_q, s_k, s_v)
//   fp8_vt_kernel     v8t      E4M3 [B, H, 128, Npad]  (V transposed, keys
//                                contiguous; columns N..Npad-1 zero), with
//                                TMA tile loads and stores
// The first two take one block of 256 threads per 64 consecutive tokens of one batch
// row; inside it a warp handles one token at a time (a half-warp per head
// row, 8 elements per lane, as in the BF16 prologue), eight heads per step
// with all of their loads issued before the arithmetic.
#pragma once

#include <cuda_fp8.h>

#include "prologue.cuh"

namespace flux {

constexpr int kQuantTokens = 64;     // tokens per block
constexpr int kQuantThreads = 256;   // 8 warps
constexpr int kQuantHeads = 8;       // heads per step of a warp (all loads of a step issued first)
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ void load_weights8(const float* w, int sub, float (&o)[8]) {
  const float4* a = reinterpret_cast<const float4*>(w + sub * 8);
  const float4 a0 = __ldg(a), a1 = __ldg(a + 1);
  o[0] = a0.x; o[1] = a0.y; o[2] = a0.z; o[3] = a0.w;
  o[4] = a1.x; o[5] = a1.y; o[6] = a1.z; o[7] = a1.w;
}

__device__ __forceinline__ float absmax8(const float (&x)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
  return m;
}

// Max over the 16 lanes of a half-warp.
__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

// 1 / scale with scale = amax / 448, or 1 when amax == 0.
__device__ __forceinline__ float inv_scale_of(uint32_t amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a > 0.f ? kE4M3Max / a : 1.f;
}

// Eight E4M3 codes of x * inv (round to nearest even, saturating), element 0 in the lowest byte.
__device__ __forceinline__ uint2 quant8(const float (&x)[8], float inv) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = __nv_cvt_float2_to_fp8x2(make_float2(x[2 * i] * inv, x[2 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

__global__ void __launch_bounds__(kQuantThreads)
    fp8_amax_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const float* __restrict__ wq,
                    const float* __restrict__ wk, TokenGeometry geo, int N, int H, float eps, RopeTable tab,
                    uint32_t* __restrict__ amax) {
  extern __shared__ uint32_t s_amax[];  // [H][3]
  const int b = blockIdx.y;
  const int n0 = blockIdx.x * kQuantTokens;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 15, half = lane >> 4;
  for (int i = threadIdx.x; i < 3 * H; i += blockDim.x) s_amax[i] = 0u;
  __syncthreads();
  float w_q[8], w_k[8];
  load_weights8(wq, sub, w_q);
  load_weights8(wk, sub, w_k);
  for (int t = warp; t < kQuantTokens; t += kQuantThreads / 32) {
    const int n = n0 + t;
    if (n >= N) break;  // warp-uniform
    float c[4], s[4];
    lane_rotation(geo, tab, n, sub, c, s);
    const size_t row0 = (static_cast<size_t>(b) * N + n) * H;
    for (int h0 = 0; h0 < H; h0 += kQuantHeads) {
      // all loads of the group first (bytes in flight), then the arithmetic
      uint4 uq[kQuantHeads / 2], uk[kQuantHeads / 2], uv[kQuantHeads / 2];
#pragma unroll
      for (int i = 0; i < kQuantHeads / 2; ++i) {
        const int h = h0 + 2 * i + half;
        uq[i] = uk[i] = uv[i] = make_uint4(0, 0, 0, 0);
        if (h < H) {
          const size_t src = (row0 + h) * kHeadDim + sub * 8;
          uq[i] = __ldg(reinterpret_cast<const uint4*>(q + src));
          uk[i] = __ldg(reinterpret_cast<const uint4*>(k + src));
          uv[i] = __ldg(reinterpret_cast<const uint4*>(v + src));
        }
      }
#pragma unroll
      for (int i = 0; i < kQuantHeads / 2; ++i) {
        const int h = h0 + 2 * i + half;
        float xq[8], xk[8], xv[8];
        unpack8(uq[i], xq);
        unpack8(uk[i], xk);
        unpack8(uv[i], xv);
        norm_rope8(xq, w_q, c, s, eps);
        norm_rope8(xk, w_k, c, s, eps);
        const float mq = half_warp_max(absmax8(xq));
        const float mk = half_warp_max(absmax8(xk));
        const float mv = half_warp_max(absmax8(xv));
        if (h < H && sub == 0) {
          atomicMax(&s_amax[3 * h + 0], __float_as_uint(mq));
          atomicMax(&s_amax[3 * h + 1], __float_as_uint(mk));
          atomicMax(&s_amax[3 * h + 2], __float_as_uint(mv));
        }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 3 * H; i += blockDim.x)
    if (s_amax[i] != 0u) atomicMax(&amax[static_cast<size_t>(b) * H * 3 + i], s_amax[i]);
}

__global__ void __launch_bounds__(kQuantThreads)
    fp8_quant_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const float* __restrict__ wq, const float* __restrict__ wk, TokenGeometry geo, int N, int H,
                     float eps,
                     RopeTable tab, const uint32_t* __restrict__ amax, uint8_t* __restrict__ q8,
                     uint8_t* __restrict__ k8, float* __restrict__ scales) {
  const int b = blockIdx.y;
  const int n0 = blockIdx.x * kQuantTokens;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 15, half = lane >> 4;
  const uint32_t* am = amax + static_cast<size_t>(b) * H * 3;

  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 3 * H; i += blockDim.x) {
      const float a = __uint_as_float(am[i]);
      scales[static_cast<size_t>(b) * H * 3 + i] = a > 0.f ? a / kE4M3Max : 1.f;
    }

  // Q', K' codes, head-major rows.
  float w_q[8], w_k[8];
  load_weights8(wq, sub, w_q);
  load_weights8(wk, sub, w_k);
  for (int t = warp; t < kQuantTokens; t += kQuantThreads / 32) {
    const int n = n0 + t;
    if (n >= N) break;  // warp-uniform
    float c[4], s[4];
    lane_rotation(geo, tab, n, sub, c, s);
    const size_t row0 = (static_cast<size_t>(b) * N + n) * H;
    for (int h0 = 0; h0 < H; h0 += kQuantHeads) {
      uint4 uq[kQuantHeads / 2], uk[kQuantHeads / 2];
#pragma unroll
      for (int i = 0; i < kQuantHeads / 2; ++i) {
        const int h = h0 + 2 * i + half;
        uq[i] = uk[i] = make_uint4(0, 0, 0, 0);
        if (h < H) {
          const size_t src = (row0 + h) * kHeadDim + sub * 8;
          uq[i] = __ldg(reinterpret_cast<const uint4*>(q + src));
          uk[i] = __ldg(reinterpret_cast<const uint4*>(k + src));
        }
      }
#pragma unroll
      for (int i = 0; i < kQuantHeads / 2; ++i) {
        const int h = h0 + 2 * i + half;
        float xq[8], xk[8];
        unpack8(uq[i], xq);
        unpack8(uk[i], xk);
        norm_rope8(xq, w_q, c, s, eps);
        norm_rope8(xk, w_k, c, s, eps);
        if (h < H) {
          const size_t dst = ((static_cast<size_t>(b) * H + h) * N + n) * kHeadDim + sub * 8;
          *reinterpret_cast<uint2*>(q8 + dst) = quant8(xq, inv_scale_of(am[3 * h + 0]));
          *reinterpret_cast<uint2*>(k8 + dst) = quant8(xk, inv_scale_of(am[3 * h + 1]));
        }
      }
    }
  }

}

// V^T codes, one 64-token x 128-dim tile of one head per CTA (128 threads):
// a TMA load brings V[b, n0 .. n0+63, h, :] into shared memory (tokens >= N
// arrive as zeros), thread d quantises head dim d of the 64 tokens into 64
// consecutive bytes of row d of the transposed tile, and one TMA store puts
// the tile at v8t[b, h, :, n0 .. n0+63] (clipped at Npad; the zero tokens
// between N and Npad become the zero padding).
constexpr int kVtTokens = 64;
constexpr int kVtThreads = 128;

__global__ void __launch_bounds__(kVtThreads)
    fp8_vt_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vt, int H,
                  const uint32_t* __restrict__ amax, uint32_t* err) {
  __shared__ __align__(128) __nv_bfloat16 vin[kVtTokens][kHeadDim];  // 16 KB
  __shared__ __align__(128) uint8_t vout[kHeadDim][kVtTokens];       // 8 KB
  __shared__ uint64_t bar;
  const int n0 = blockIdx.x * kVtTokens;
  const int bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int d = threadIdx.x;
  if (d == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (d == 0) {
    mbar_arrive_expect_tx(&bar, sizeof(vin));
    tma_load_4d(smem_u32(vin), &tm_v, &bar, 0, h, n0, b);
  }
  // bounded wait on the load (every thread); a timeout leaves the tile unwritten
  const uint32_t ba = smem_u32(&bar);
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;
  while (!mbar_try_wait(ba, 0))
    if (globaltimer_ns() - t0 > kWaitLimitNs) { ok = false; break; }
  if (__syncthreads_or(!ok)) {
    if (d == 0) atomicOr(err, kErrTimeout);
    // the copy may still land: keep the shared memory alive until it has (bounded)
    const uint64_t t1 = globaltimer_ns();
    while (!mbar_try_wait(ba, 0) && globaltimer_ns() - t1 < kWaitLimitNs) {}
    return;
  }
  const float inv = inv_scale_of(amax[3 * bh + 2]);
  uint32_t w[kVtTokens / 4];
#pragma unroll
  for (int t = 0; t < kVtTokens; t += 4) {
    const float x0 = __bfloat162float(vin[t][d]) * inv, x1 = __bfloat162float(vin[t + 1][d]) * inv;
    const float x2 = __bfloat162float(vin[t + 2][d]) * inv, x3 = __bfloat162float(vin[t + 3][d]) * inv;
    w[t / 4] = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3) |
               (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x2, x3), __NV_SATFINITE, __NV_E4M3))
                << 16);
  }
#pragma unroll
  for (int c = 0; c < kVtTokens / 16; ++c)
    reinterpret_cast<uint4*>(vout[d])[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (d == 0) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(&tm_vt)),
                 "r"(smem_u32(vout)), "r"(n0), "r"(0), "r"(bh)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

}  // namespace flux
