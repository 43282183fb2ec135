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
// Four kernels over q, k, v (bf16 [B, N, H, 128]); amax (fp32 bit patterns,
// [B*H][3] for Q', K', V; positive floats order like their bits, so atomicMax
// on the bits is a float max) must be zero on entry:
//   fp8_vamax_kernel                  |V| max, TMA tiles of 64 tokens of a head
//   qk_norm_rope_kernel<AmaxRows>     the BF16 prologue's stream kernel with
//                                     the rows reduced to |Q'|, |K'| maxima
//                                     instead of stored
//   qk_norm_rope_kernel<E4m3Rows>     the same rows again, written as E4M3
//                                       q8, k8   [B, H, N, 128]
//                                       scales   fp32 [B, H, 3] = (s_q, s_k, s_v)
//   fp8_vt_kernel                     v8t E4M3 [B, H, 128, Npad] (V transposed,
//                                     keys contiguous; columns N..Npad-1 zero;
//                                     the keys of every 8 in the order
//                                     0 2 4 6 1 3 5 7 of the attention's P.V)
// Recomputing Q', K' in the second pass costs less than a round trip of an
// fp32 or bf16 copy through HBM, and keeps a single rounding, fp32 -> E4M3.
#pragma once

#include <cuda_fp8.h>

#include "prologue.cuh"

namespace flux {

constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float absmax8(const float (&x)[8]) {
  return fmax3(fmax3(fabsf(x[0]), fabsf(x[1]), fabsf(x[2])), fmax3(fabsf(x[3]), fabsf(x[4]), fabsf(x[5])),
               fmaxf(fabsf(x[6]), fabsf(x[7])));
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

// Output policy of the stream kernel: per-(b, h) amax of Q' and K'.  Each
// lane keeps its running |max| of every (tensor, head) row it owns in its
// own shared-memory slot ([2][H][16] per warp; a slot has one writer, so no
// atomics), and folds the slots into the global amax with one atomicMax per
// (tensor, head) whenever the warp's batch row changes and after its last
// token.
struct AmaxRows {
  static constexpr int kParts = 2;  // half tokens, twelve warps: more warps to hide latency, as
  static constexpr int kStages = 2;
  static constexpr int kWarps = 12; // nothing (or only codes, below) is written per row
  static constexpr int kPairs = 3;  // six independent rows per half-warp
  uint32_t* amax;  // [B*H][3]
  float* slot;
  int H, cur_b;
  static __host__ __device__ constexpr int warp_scratch(int H) { return 2 * H * 16 * static_cast<int>(sizeof(float)); }
  __device__ __forceinline__ void init(uint8_t* scratch, int, int heads) {
    H = heads;
    cur_b = -1;
    slot = reinterpret_cast<float*>(scratch) + static_cast<size_t>(threadIdx.x >> 5) * 2 * H * 16;
    for (int i = threadIdx.x & 31; i < 2 * H * 16; i += 32) slot[i] = 0.f;
    __syncwarp();
  }
  __device__ void flush() {
    __syncwarp();
    for (int i = threadIdx.x & 31; i < 2 * H; i += 32) {  // i = t H + h
      float m = 0.f;
#pragma unroll 4
      for (int l = 0; l < 16; ++l) {
        m = fmaxf(m, slot[i * 16 + l]);
        slot[i * 16 + l] = 0.f;
      }
      const int t = i / H, h = i - t * H;
      if (m > 0.f) atomicMax(&amax[(static_cast<size_t>(cur_b) * H + h) * 3 + t], __float_as_uint(m));
    }
    __syncwarp();
  }
  __device__ __forceinline__ void token(int b) {
    if (b != cur_b) {
      if (cur_b >= 0) flush();
      cur_b = b;
    }
  }
  __device__ __forceinline__ void row(int t, int, int h, size_t, const float (&x)[8], bool valid) {
    if (!valid) return;
    float* p = slot + (t * H + h) * 16 + (threadIdx.x & 15);
    *p = fmaxf(*p, absmax8(x));
  }
  __device__ __forceinline__ void finish() {
    if (cur_b >= 0) flush();
  }
};

// The values two E4M3 codes stand for (c16: two codes, the first in the low byte).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t c16) {
  return __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c16), __NV_E4M3)));
}

// Squared quantisation error sum_i (x_i - code_i * s)^2 of eight values and their codes.
__device__ __forceinline__ float sq_error8(const float (&x)[8], uint2 c, float s) {
  const uint32_t w[4] = {c.x & 0xFFFFu, c.x >> 16, c.y & 0xFFFFu, c.y >> 16};
  float e = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 d = e4m3x2_to_float2(w[i]);
    const float r0 = x[2 * i] - d.x * s, r1 = x[2 * i + 1] - d.y * s;
    e = fmaf(r0, r0, e);
    e = fmaf(r1, r1, e);
  }
  return e;
}

// Output policy of the stream kernel: E4M3 codes of Q' / s_q and K' / s_k,
// head-major; block 0 also writes the scales of all three tensors.  With
// errk set (VC-Attention repair) it also writes, per (b, h, token), the
// squared quantisation error |k' - code s_k|^2 of the K' row, summed by the
// half-warp that holds the row in a fixed order.
struct E4m3Rows {
  static constexpr int kParts = 2;
  static constexpr int kStages = 2;
  static constexpr int kWarps = 12;
  static constexpr int kPairs = 3;
  uint8_t* q8;
  uint8_t* k8;
  const uint32_t* amax;  // [B*H][3], complete
  float* scales;         // [B*H][3]
  int H, n_scales;
  float* errk;           // [B*H][N] or nullptr
  static __host__ __device__ constexpr int warp_scratch(int) { return 0; }
  __device__ __forceinline__ void init(uint8_t*, int, int) {
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < n_scales; i += blockDim.x) {
        const float a = __uint_as_float(amax[i]);
        scales[i] = a > 0.f ? a / kE4M3Max : 1.f;
      }
  }
  __device__ __forceinline__ void token(int) {}
  __device__ __forceinline__ void row(int t, int b, int h, size_t dst, const float (&x)[8], bool valid) {
    const uint32_t a = __ldg(amax + (static_cast<size_t>(b) * H + h) * 3 + t);
    const uint2 c = quant8(x, inv_scale_of(a));
    if (valid) *reinterpret_cast<uint2*>((t == 0 ? q8 : k8) + dst) = c;
    if (errk != nullptr && t == 1) {  // warp-uniform: every lane shuffles
      const float af = __uint_as_float(a);
      float e = sq_error8(x, c, af > 0.f ? af / kE4M3Max : 1.f);
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) e += __shfl_xor_sync(0xFFFFFFFFu, e, off);
      // dst / 128 = (b H + h) N + n: the row's token index in [B*H][N]
      if (valid && (threadIdx.x & 15) == 0) errk[dst >> 7] = e;
    }
  }
  __device__ __forceinline__ void finish() {}
};

// One 64-token x 128-dim bf16 tile of V (tokens >= N arrive as zeros) into
// shared memory by TMA, with a bounded wait on every thread.  Returns false
// (after the copy has landed or the second bounded wait ended) when the wait
// ran out; the error word is set then.
constexpr int kVtTokens = 64;
constexpr int kVtThreads = 128;

__device__ __forceinline__ bool v_tile_load(const CUtensorMap* tm_v, __nv_bfloat16 (*vin)[kHeadDim], uint64_t* bar,
                                            int h, int n0, int b, uint32_t* err) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, kVtTokens * kHeadDim * 2);
    tma_load_4d(smem_u32(vin), tm_v, bar, 0, h, n0, b);
  }
  const uint32_t ba = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;
  while (!mbar_try_wait(ba, 0))
    if (globaltimer_ns() - t0 > kWaitLimitNs) { ok = false; break; }
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
    // the copy may still land: keep the shared memory alive until it has (bounded)
    const uint64_t t1 = globaltimer_ns();
    while (!mbar_try_wait(ba, 0) && globaltimer_ns() - t1 < kWaitLimitNs) {}
    return false;
  }
  return true;
}

// |V| max of one 64-token tile of one head per CTA: thread d takes head dim
// d, then a block max and one atomicMax into amax[b*H + h][2].
__global__ void __launch_bounds__(kVtThreads)
    fp8_vamax_kernel(const __grid_constant__ CUtensorMap tm_v, int H, uint32_t* __restrict__ amax, uint32_t* err) {
  __shared__ __align__(128) __nv_bfloat16 vin[kVtTokens][kHeadDim];  // 16 KB
  __shared__ uint64_t bar;
  __shared__ float wmax[kVtThreads / 32];
  const int bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  if (!v_tile_load(&tm_v, vin, &bar, h, blockIdx.x * kVtTokens, b, err)) return;
  const int d = threadIdx.x;
  float m = 0.f;
#pragma unroll 16
  for (int t = 0; t < kVtTokens; ++t) m = fmaxf(m, fabsf(__bfloat162float(vin[t][d])));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((d & 31) == 0) wmax[d >> 5] = m;
  __syncthreads();
  if (d == 0) {
    m = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    if (m > 0.f) atomicMax(&amax[3 * bh + 2], __float_as_uint(m));
  }
}

// V^T codes, one 64-token x 128-dim tile of one head per CTA (128 threads):
// a TMA load brings V[b, n0 .. n0+63, h, :] into shared memory (tokens >= N
// arrive as zeros), thread d quantises head dim d of the 64 tokens into 64
// consecutive bytes of row d of the transposed tile, and one TMA store puts
// the tile at v8t[b, h, :, n0 .. n0+63] (clipped at Npad; the zero tokens
// between N and Npad become the zero padding).
//
// MMA_ORDER: within every 8 tokens the columns hold tokens 0, 2, 4, 6, 1, 3,
// 5, 7 -- the key order of the P.V MMA in the FP8 attention, whose softmax
// threads hold the even or the odd keys of a row (attention.cuh).  Tiles
// start at multiples of 64 tokens, so the groups of 8 are those of the key
// blocks, and Npad (a multiple of 16) never splits one.
//
// With errv set (VC-Attention repair) the kernel also writes, per token of
// the tile, the squared quantisation error |v - code s_v|^2 of its V row:
// thread d holds dim d of the 64 tokens, a butterfly over the lanes leaves
// lane l of warp w with the sums over its 32 dims of tokens 2l and 2l + 1,
// and thread t < 64 adds the four warps' sums of token t, in a fixed order.
template <bool MMA_ORDER>
__global__ void __launch_bounds__(kVtThreads)
    fp8_vt_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vt, int H,
                  const uint32_t* __restrict__ amax, uint32_t* err, float* __restrict__ errv, int N) {
  __shared__ __align__(128) __nv_bfloat16 vin[kVtTokens][kHeadDim];  // 16 KB
  __shared__ __align__(128) uint8_t vout[kHeadDim][kVtTokens];       // 8 KB
  __shared__ uint64_t bar;
  const int n0 = blockIdx.x * kVtTokens;
  const int bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int d = threadIdx.x;
  if (!v_tile_load(&tm_v, vin, &bar, h, n0, b, err)) return;
  // x / scale = 448 x / amax, rounded once, as the exact quotient would be:
  // with amax = d 2^E, d in [1, 2), the numerator a = 448 (2^-E x) is exact
  // for a bf16 x (<= 896, or tiny enough to give code 0), and the quotient
  // a / d comes from q0 = a rcp(d) with Markstein's correction
  // q = q0 + (a - q0 d) rcp(d) (residual exact by FMA).  A product with a
  // rounded 1 / scale alone misses the code decision when x / scale is a
  // midpoint between two codes, which bf16 V with amax like 24.5 hits often.
  // The sign of x is copied onto the quotient, so that a negative x whose
  // 2^-E x underflows still gives the code of -0.
  const float am = __uint_as_float(amax[3 * bh + 2]);
  float den = am > 0.f ? am : kE4M3Max;  // scale 1 when amax == 0
  const float pre = den < 1.17549435e-38f ? 16777216.f : 1.f;  // subnormal amax: x and amax times 2^24 first
  den *= pre;
  const int ex = static_cast<int>((__float_as_uint(den) >> 23) & 0xFFu) - 127;
  const float dm = __uint_as_float((__float_as_uint(den) & 0x007FFFFFu) | 0x3F800000u);
  const float s2 = ldexpf(1.f, -ex);
  const float y = __frcp_rn(dm);
  auto code_value = [&](float v) {
    const float a = ((v * pre) * s2) * kE4M3Max;
    const float q0 = a * y;
    return copysignf(fmaf(fmaf(-q0, dm, a), y, q0), v);  // keeps -0 for a negative x that underflows
  };
  uint32_t w[kVtTokens / 4];
#pragma unroll
  for (int i = 0; i < kVtTokens / 4; ++i) {
    // byte b of word i: token 4i + b, or (MMA_ORDER) 8 (i / 2) + i % 2 + 2b
    const int t = MMA_ORDER ? 8 * (i >> 1) + (i & 1) : 4 * i;
    const int st = MMA_ORDER ? 2 : 1;
    const float x0 = code_value(__bfloat162float(vin[t][d]));
    const float x1 = code_value(__bfloat162float(vin[t + st][d]));
    const float x2 = code_value(__bfloat162float(vin[t + 2 * st][d]));
    const float x3 = code_value(__bfloat162float(vin[t + 3 * st][d]));
    w[i] = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3) |
           (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x2, x3), __NV_SATFINITE, __NV_E4M3))
            << 16);
  }
  if (errv != nullptr) {  // block-uniform
    __shared__ float wsum[kVtThreads / 32][kVtTokens];
    const float sv = am > 0.f ? am / kE4M3Max : 1.f;
    float e[kVtTokens];  // by token
#pragma unroll
    for (int i = 0; i < kVtTokens / 4; ++i) {
      const int t = MMA_ORDER ? 8 * (i >> 1) + (i & 1) : 4 * i;  // token of byte 0 of word i
      const int st = MMA_ORDER ? 2 : 1;
      const float2 a = e4m3x2_to_float2(w[i] & 0xFFFFu), c = e4m3x2_to_float2(w[i] >> 16);
      const float r0 = __bfloat162float(vin[t][d]) - a.x * sv;
      const float r1 = __bfloat162float(vin[t + st][d]) - a.y * sv;
      const float r2 = __bfloat162float(vin[t + 2 * st][d]) - c.x * sv;
      const float r3 = __bfloat162float(vin[t + 3 * st][d]) - c.y * sv;
      e[t] = r0 * r0;
      e[t + st] = r1 * r1;
      e[t + 2 * st] = r2 * r2;
      e[t + 3 * st] = r3 * r3;
    }
    // butterfly: at offset o a lane keeps the half of its tokens its bit o selects
    const int lane = d & 31;
#pragma unroll
    for (int o = 16, n = kVtTokens / 2; o >= 1; o >>= 1, n >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float keep = up ? e[i + n] : e[i];
        const float give = up ? e[i] : e[i + n];
        e[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, o);
      }
    }
    wsum[d >> 5][2 * lane] = e[0];
    wsum[d >> 5][2 * lane + 1] = e[1];
    __syncthreads();
    if (d < kVtTokens && n0 + d < N)
      errv[static_cast<size_t>(bh) * N + n0 + d] = ((wsum[0][d] + wsum[1][d]) + wsum[2][d]) + wsum[3][d];
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

// E4M3 codes of bf16 Q', K' (head-major [B*H][N][128], as the QKV projection
// writes them) with the per-(b, h) scales of amax ([B*H][3], complete); each
// thread step turns 16 values (two 16-byte loads) into one 16-byte store.
// Block 0 also writes the three scales of every head.
constexpr int kCodesThreads = 256;

__global__ void __launch_bounds__(kCodesThreads)
    fp8_codes_kernel(const __nv_bfloat16* __restrict__ qn, const __nv_bfloat16* __restrict__ kn, int N, int BH,
                     const uint32_t* __restrict__ amax, uint8_t* __restrict__ q8, uint8_t* __restrict__ k8,
                     float* __restrict__ scales) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 3 * BH; i += blockDim.x) {
      const float a = __uint_as_float(amax[i]);
      scales[i] = a > 0.f ? a / kE4M3Max : 1.f;
    }
  const size_t per_head = static_cast<size_t>(N) * kHeadDim / 16;  // 16-value items of one head
  const size_t items = 2 * static_cast<size_t>(BH) * per_head;
  for (size_t it = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
       it += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = it >= static_cast<size_t>(BH) * per_head;  // 0: Q', 1: K'
    const size_t j = it - t * static_cast<size_t>(BH) * per_head;
    const int bh = static_cast<int>(j / per_head);
    const float inv = inv_scale_of(__ldg(amax + 3 * bh + t));
    const uint4* src = reinterpret_cast<const uint4*>(t == 0 ? qn : kn) + 2 * j;
    float x[8], y[8];
    unpack8(__ldg(src), x);
    unpack8(__ldg(src + 1), y);
    const uint2 a = quant8(x, inv), c = quant8(y, inv);
    reinterpret_cast<uint4*>(t == 0 ? q8 : k8)[j] = make_uint4(a.x, a.y, c.x, c.y);
  }
}

}  // namespace flux
