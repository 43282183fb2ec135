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

// (cos, sin) of pos * freq_j for the positions 0 .. kRotPositions-1 and all
// 64 pairs, [pos][j], computed once per handle (rot_table_kernel) with the
// same sincosf as the direct path below, so the two give the same bits.  The
// [text | image | reference] geometries of FLUX stay inside it up to 4096
// pixels a side (256 patches); other positions take the direct path.
constexpr int kRotPositions = 256;

__global__ void rot_table_kernel(RopeTable tab, float2* __restrict__ rot) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= kRotPositions * (kHeadDim / 2)) return;
  const int pos = i / (kHeadDim / 2), j = i - pos * (kHeadDim / 2);
  float s, c;
  sincosf(static_cast<float>(pos) * tab.freq[j], &s, &c);
  rot[i] = make_float2(c, s);
}

// Rotation angles of the four pairs a lane owns (pairs 4 sub .. 4 sub + 3):
// from the table when rot is set and the position is in it, else sincosf.
// The axis of a pair picks its position id with selects, not an indexed
// local array.
__device__ __forceinline__ void lane_rotation(const TokenGeometry& geo, const RopeTable& tab, const float2* rot,
                                              int n, int sub, float (&c)[4], float (&s)[4]) {
  int p[3];
  token_position(geo, n, p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = sub * 4 + i;
    const int a = tab.axis[j];
    const int pos = a == 0 ? p[0] : (a == 1 ? p[1] : p[2]);
    if (rot != nullptr && static_cast<unsigned>(pos) < static_cast<unsigned>(kRotPositions)) {
      const float2 cs = __ldg(rot + pos * (kHeadDim / 2) + j);
      c[i] = cs.x;
      s[i] = cs.y;
    } else {
      sincosf(static_cast<float>(pos) * tab.freq[j], &s[i], &c[i]);
    }
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

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

// Per-lane coefficients of the weighted rotation.  With r the row's
// reciprocal RMS, the weight w and the rotation (c, s) of pair (x0, x1) fold
// into
//   out0 = r (x0 w0 c - x1 w1 s),   out1 = r (x0 w0 s + x1 w1 c),
// computed two pairs at a time in packed fp32x2 operations: lane pairs
// (0, 1) and (2, 3) of its four, the even elements (x0 of each pair) in one
// operand and the odd ones in the other.  m = 0, 1 picks the pair of pairs.
struct RotCoef {
  float a[4], b[4], c[4], d[4];  // [2m + e]: w0 c, -w1 s, w0 s, w1 c of pair 2m + e
};

__device__ __forceinline__ void rot_coef(const float (&w)[8], const float (&c)[4], const float (&s)[4],
                                         RotCoef& k) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    k.a[i] = w[2 * i] * c[i];
    k.b[i] = -w[2 * i + 1] * s[i];
    k.c[i] = w[2 * i] * s[i];
    k.d[i] = w[2 * i + 1] * c[i];
  }
}

// RMSNorm, weight and rotation of the 8 elements a lane holds (a half-warp
// holds the row), in packed fp32x2 arithmetic.
__device__ __forceinline__ void norm_rope8_packed(float (&x)[8], const RotCoef& k, float eps) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    fma2(s0, s1, x[4 * m], x[4 * m + 2], x[4 * m], x[4 * m + 2], s0, s1);
    fma2(s0, s1, x[4 * m + 1], x[4 * m + 3], x[4 * m + 1], x[4 * m + 3], s0, s1);
  }
  float ss = s0 + s1;
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float r = rsqrtf(ss * (1.0f / kHeadDim) + eps);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const float e0 = x[4 * m], e1 = x[4 * m + 2];      // x0 of pairs 2m, 2m + 1
    const float o0 = x[4 * m + 1], o1 = x[4 * m + 3];  // x1 of pairs 2m, 2m + 1
    float u0, u1, v0, v1;
    mul2(u0, u1, o0, o1, k.b[2 * m], k.b[2 * m + 1]);
    fma2(u0, u1, e0, e1, k.a[2 * m], k.a[2 * m + 1], u0, u1);
    mul2(v0, v1, o0, o1, k.d[2 * m], k.d[2 * m + 1]);
    fma2(v0, v1, e0, e1, k.c[2 * m], k.c[2 * m + 1], v0, v1);
    mul2(x[4 * m], x[4 * m + 2], u0, u1, r, r);
    mul2(x[4 * m + 1], x[4 * m + 3], v0, v1, r, r);
  }
}

// Streaming layout: a persistent block per SM of W warps, each streaming its
// own tokens through its own S-stage ring.  Warp w of block x takes tokens
// t = W x + w, then every W * gridDim.x-th, in P parts of ceil(H / P) heads:
// a stage holds one part (its q rows and its k rows, two bulk copies of
// contiguous bytes, since a token's heads are adjacent in [B, N, H, 128]).
// Lane 0 keeps the next S - 1 parts in flight and refills a stage as soon as
// the warp has read it; no warp waits for another.  Per token the warp
// computes (b, n), the (cos, sin) pairs and the rotation coefficients once,
// then normalises, rotates and stores the head rows of each part (a
// half-warp per row, read from shared memory, written head-major).
constexpr int kProMaxWarps = 16;                     // warps per block at most (any output policy)
constexpr int kProStages = 2;                        // parts per warp ring of whole tokens (Bf16Rows)
constexpr int kProSmemBytes = 220 * 1024;            // rings and the output policy's scratch
constexpr int kProRingBytes = 192 * 1024;            // bounds H: one warp's two whole-token stages fit
constexpr int kProRowBytes = 2 * kHeadDim * 2;       // one head row of q and one of k
constexpr int kProMaxHeads = kProRingBytes / (kProStages * kProRowBytes);  // 192: one warp, whole tokens

// Heads per part when a token is cut into `parts` parts.
__host__ __device__ constexpr int prologue_part_heads(int H, int parts) { return (H + parts - 1) / parts; }

// Shared memory of one warp: its ring of `stages` parts and its scratch.
__host__ __device__ constexpr int prologue_warp_bytes(int H, int parts, int stages, int scratch) {
  return stages * kProRowBytes * prologue_part_heads(H, parts) + scratch;
}

// Warps per block (1 .. max_warps) for H heads in `parts` parts, rings of
// `stages` parts and `scratch` bytes of policy scratch per warp (H <=
// kProMaxHeads: every policy fits one warp then, checked in the kernel).
__host__ __device__ constexpr int prologue_warps(int H, int parts, int stages, int max_warps, int scratch) {
  return kProSmemBytes / prologue_warp_bytes(H, parts, stages, scratch) < max_warps
             ? kProSmemBytes / prologue_warp_bytes(H, parts, stages, scratch)
             : max_warps;
}

// What the stream kernel does with the normalised, rotated rows.  Every
// output policy has
//   warp_scratch(H)             shared memory per warp it needs after the rings
//   init(scratch, W, H)         once per warp (all lanes), before the first token
//   token(b)                    warp-uniform, at every token (b its batch row)
//   row(t, b, h, dst, x, valid) one lane's 8 values of row h of tensor t (0: Q',
//                               1: K'); dst = element offset of those 8 values in
//                               a head-major [B, H, N, 128] tensor.  Called by
//                               all 32 lanes together (warp-uniform); a half-warp
//                               past the part's last head has valid == false,
//                               zeros in x, and must store nothing
//   finish()                    once per warp (all lanes), after the last token
// and its stream shape: kParts parts per token, kStages parts per warp
// ring, kWarps warps per block at most (the rings' shared memory may allow
// fewer), kPairs head pairs a warp
// works on at a time.
// The BF16 policy writes Q', K' bf16 [B, H, N, 128].  Whole tokens and eight
// warps: with twice the bytes written per row, more and smaller parts lost.
struct Bf16Rows {
  static constexpr int kParts = 1;
  static constexpr int kStages = kProStages;
  static constexpr int kWarps = 8;
  static constexpr int kPairs = 2;
  __nv_bfloat16* qn;
  __nv_bfloat16* kn;
  static __host__ __device__ constexpr int warp_scratch(int) { return 0; }
  __device__ __forceinline__ void init(uint8_t*, int, int) {}
  __device__ __forceinline__ void token(int) {}
  __device__ __forceinline__ void row(int t, int, int, size_t dst, const float (&x)[8], bool valid) {
    if (valid) *reinterpret_cast<uint4*>((t == 0 ? qn : kn) + dst) = pack8(x);
  }
  __device__ __forceinline__ void finish() {}
};

struct StreamArgs {
  const __nv_bfloat16* q;  // [B, N, H, 128]
  const __nv_bfloat16* k;
  const float* wq;         // [128] RMSNorm weights
  const float* wk;
  TokenGeometry geo;
  int B, N, H;
  float eps;
  RopeTable tab;
  uint32_t* err;
  const float2* rot = nullptr;  // rotation table (kRotPositions x 64), or none
};

// Launch shape of the stream kernel for output policy Out and H heads.
template <class Out>
__host__ __device__ constexpr int stream_warps(int H) {
  return prologue_warps(H, Out::kParts, Out::kStages, Out::kWarps, Out::warp_scratch(H));
}
template <class Out>
__host__ __device__ constexpr size_t stream_smem(int H) {
  return static_cast<size_t>(stream_warps<Out>(H)) *
         prologue_warp_bytes(H, Out::kParts, Out::kStages, Out::warp_scratch(H));
}

template <class Out>
__global__ void __launch_bounds__(32 * Out::kWarps, 1) qk_norm_rope_kernel(const StreamArgs a, Out out) {
  static_assert(Out::kWarps <= kProMaxWarps, "barrier array");
  static_assert(prologue_warp_bytes(kProMaxHeads, Out::kParts, Out::kStages, Out::warp_scratch(kProMaxHeads)) <=
                    kProSmemBytes,
                "one warp's ring and scratch fit at the largest head count");
  // Every CTA of this grid is resident at once (grid <= SMs, one block per
  // SM): the attention kernel after it may be scheduled now and set up on
  // SMs whose block has finished.
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t ring[];  // [W][S][q rows | k rows] of one part; then Out's scratch
  __shared__ uint64_t full[Out::kWarps][Out::kStages];  // per warp: stage s holds a part
  __shared__ int abort_flag;
  const int W = blockDim.x >> 5;
  constexpr int S = Out::kStages;
  const int H = a.H, N = a.N;
  const int hs = Out::kParts == 1 ? H : prologue_part_heads(H, Out::kParts);
  const int P = Out::kParts == 1 ? 1 : (H + hs - 1) / hs;  // parts of a token (<= kParts, none empty)
  const uint32_t srow = static_cast<uint32_t>(hs) * kHeadDim * 2;  // q (or k) bytes of a full part
  const long long tokens = static_cast<long long>(a.B) * N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* ab = &abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[warp][s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  uint8_t* wring = ring + static_cast<size_t>(warp) * S * 2 * srow;
  const long long first = static_cast<long long>(blockIdx.x) * W + warp;
  const long long step = static_cast<long long>(gridDim.x) * W;
  // Part u of the warp's stream: token first + (u / P) step, heads from (u % P) hs.
  auto issue = [&](int u, int s) {
    const long long t = first + static_cast<long long>(u / P) * step;
    if (t >= tokens) return;
    const int h0 = (u % P) * hs;
    const uint32_t bytes = static_cast<uint32_t>(min(hs, H - h0)) * kHeadDim * 2;
    const size_t off = (static_cast<size_t>(t) * H + h0) * kHeadDim;
    mbar_arrive_expect_tx(&full[warp][s], 2 * bytes);
    bulk_load(smem_u32(wring + s * 2 * srow), a.q + off, bytes, &full[warp][s]);
    bulk_load(smem_u32(wring + s * 2 * srow + srow), a.k + off, bytes, &full[warp][s]);
  };
  if (lane == 0)  // the warp's first S parts
    for (int u = 0; u < S; ++u) issue(u, u);
  out.init(ring + static_cast<size_t>(W) * S * 2 * srow, W, H);
  const int sub = lane & 15;
  const int half = lane >> 4;
  float w_q[8], w_k[8];
  {
    const float4* pa = reinterpret_cast<const float4*>(a.wq + sub * 8);
    const float4* pb = reinterpret_cast<const float4*>(a.wk + sub * 8);
    const float4 a0 = __ldg(pa), a1 = __ldg(pa + 1), b0 = __ldg(pb), b1 = __ldg(pb + 1);
    w_q[0] = a0.x; w_q[1] = a0.y; w_q[2] = a0.z; w_q[3] = a0.w;
    w_q[4] = a1.x; w_q[5] = a1.y; w_q[6] = a1.z; w_q[7] = a1.w;
    w_k[0] = b0.x; w_k[1] = b0.y; w_k[2] = b0.z; w_k[3] = b0.w;
    w_k[4] = b1.x; w_k[5] = b1.y; w_k[6] = b1.z; w_k[7] = b1.w;
  }
  const size_t head_stride = static_cast<size_t>(N) * kHeadDim;  // elements between heads of Q' / K'
  int u = 0;
  bool aborted = false;
  RotCoef kq, kk;
  int b = 0, n = 0;
  for (long long t = first; t < tokens; t += step) {
    for (int p = 0; p < P; ++p, ++u) {
      const int s = u % S;
      const bool ok = mbar_wait(&full[warp][s], (u / S) & 1, ab, a.err);
      if (__any_sync(0xFFFFFFFFu, !ok)) { aborted = true; break; }
      if (p == 0) {
        b = static_cast<int>(t / N);
        n = static_cast<int>(t - static_cast<long long>(b) * N);
        out.token(b);
        float cs[4], sn[4];
        lane_rotation(a.geo, a.tab, a.rot, n, sub, cs, sn);
        rot_coef(w_q, cs, sn, kq);
        rot_coef(w_k, cs, sn, kk);
      }
      const int h0 = p * hs;
      const int h1 = min(H, h0 + hs);
      const uint8_t* sq = wring + s * 2 * srow + sub * 16;  // row h of the part at (h - h0) 256 bytes
      const size_t dst = (static_cast<size_t>(b) * H * N + n) * kHeadDim + sub * 8;
      // kPairs head pairs per step: 2 kPairs independent rows per half-warp,
      // so that their shuffle reductions overlap.  A half-warp past the
      // part's last head computes on zeros and stores nothing.
      constexpr int kProPairs = Out::kPairs;
      for (int hp = h0; hp < h1; hp += 2 * kProPairs) {
        uint4 uq[kProPairs], uk[kProPairs];
#pragma unroll
        for (int i = 0; i < kProPairs; ++i) {
          const int h = hp + 2 * i + half;
          uq[i] = uk[i] = make_uint4(0, 0, 0, 0);
          if (h < h1) {
            uq[i] = *reinterpret_cast<const uint4*>(sq + (h - h0) * kHeadDim * 2);
            uk[i] = *reinterpret_cast<const uint4*>(sq + srow + (h - h0) * kHeadDim * 2);
          }
        }
        float xq[kProPairs][8], xk[kProPairs][8];
#pragma unroll
        for (int i = 0; i < kProPairs; ++i) {
          unpack8(uq[i], xq[i]);
          unpack8(uk[i], xk[i]);
        }
#pragma unroll
        for (int i = 0; i < kProPairs; ++i) {
          norm_rope8_packed(xq[i], kq, a.eps);
          norm_rope8_packed(xk[i], kk, a.eps);
        }
#pragma unroll
        for (int i = 0; i < kProPairs; ++i) {
          const int h = hp + 2 * i + half;
          const bool valid = h < h1;
          const int hv = valid ? h : h0;
          out.row(0, b, hv, dst + hv * head_stride, xq[i], valid);
          out.row(1, b, hv, dst + hv * head_stride, xk[i], valid);
        }
      }
      __syncwarp();  // every lane has read the stage: refill it with part u + S
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(u + S, s);
      }
    }
    if (aborted) break;
  }
  if (aborted) {
    if (lane == 0)  // loads still in flight must land before the block exits (bounded)
      for (int uu = u; uu < u + S; ++uu) {
        if (first + static_cast<long long>(uu / P) * step >= tokens) break;
        const uint32_t ba = smem_u32(&full[warp][uu % S]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(ba, (uu / S) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    return;
  }
  out.finish();
}

}  // namespace flux
