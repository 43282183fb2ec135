// flux_attn.cu -- C ABI of the joint text/image attention library (see
// include/flux_attn.h for the contract of every entry point).
//
// Host side only: argument checks, workspace, TMA tensor maps and launches.
// The arithmetic of the path runs in the kernels of prologue.cuh,
// quantize_fp8.cuh and attention.cuh.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "flux_attn.h"
#include "attention.cuh"
#include "prologue.cuh"
#include "qkv_gemm.cuh"
#include "quantize_fp8.cuh"
#include "sol_sparse.cuh"
#include "vc_repair.cuh"

struct flux_attn {
  flux_attn_config cfg;
  int device;
  int num_sms;
  size_t ws_bytes;
  void* ws;               // one allocation, carved below
  __nv_bfloat16* qn;      // BF16: [B, H, max_tokens, 128]
  __nv_bfloat16* kn;      // BF16: [B, H, max_tokens, 128]
  __nv_bfloat16* vw;      // BF16: [B, max_tokens, H, 128], V of flux_attn_forward_hidden
  uint8_t* q8;            // FP8: E4M3 [B, H, max_tokens, 128]
  uint8_t* k8;            // FP8: E4M3 [B, H, max_tokens, 128]
  uint8_t* v8t;           // FP8: E4M3 [B, H, 128, pad16(max_tokens)]
  uint32_t* amax;         // FP8: [B, H, 3] fp32 bits
  float* scales;          // FP8: [B, H, 3]
  float2* rope;           // BF16: (cos, sin) table [max_tokens][64] of the QKV projection
  float2* rot;            // (cos, sin) per position [kRotPositions][64], built at creation
  float* errk;            // VC: K' quantisation error per token [B*H][max_tokens]
  float* errv;            // VC: V quantisation error per token [B*H][max_tokens]
  int32_t* sel;           // VC: repaired tokens [B*H][r_max]
  __nv_bfloat16* krep;    // VC: k' / s_k of the repaired tokens [B*H][r_max][128]
  __nv_bfloat16* vrep;    // VC: v / s_v of the repaired tokens [B*H][r_max][128]
  int r_max;              // VC: ceil(rho max_tokens)
  float* qbar;            // SOL: block means of Q' [B*H][nb_max][128]
  float* kbar;            // SOL: block means of K' [B*H][nb_max][128]
  uint8_t* keep;          // SOL: block mask [B*H][nb][nb] of the last forward
  uint16_t* sol_list;     // SOL: key-block lists [B*H][ncta][nb]
  int* sol_count;         // SOL: list lengths [B*H][ncta]
  uint32_t* err;          // device error word
  flux::RopeTable rope_tab;
};

namespace {

thread_local std::string g_last_error;

// Sol-Attention's block mask holds nb^2 bytes per head (nb = max_tokens / 128),
// and its keep kernel scores at most flux::sol::kMaxNb blocks.
constexpr int kSolMaxTokens = flux::sol::kMaxNb * flux::sol::kBlock;

// An NVTX range over the host-side enqueue of one call or one kernel launch:
// profilers (Nsight Systems, ncu --nvtx) show the library's steps by name.
// Header-only NVTX v3; without an attached tool each push / pop is a branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(FLUX_ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Driver entry points, fetched through the runtime so the library does not
// link libcuda directly.
struct Driver {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  PFN_cuPointerGetAttribute_v4000 ptr_attr = nullptr;
};

const Driver& driver() {
  static Driver d;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.ptr_attr = reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(p);
  });
  return d;
}

// A device buffer argument: non-null, 16-byte aligned, device memory, and the
// allocation it belongs to covers [p, p + bytes).
int check_buffer(const void* p, size_t bytes, const char* name) {
  if (p == nullptr) return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) & 15u)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  const Driver& d = driver();
  if (d.ptr_attr == nullptr) return fail(FLUX_ATTN_ERR_CUDA, "cuPointerGetAttribute unavailable");
  CUdeviceptr start = 0;
  size_t size = 0;
  unsigned int mem_type = 0;
  const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(p);
  if (d.ptr_attr(&mem_type, CU_POINTER_ATTRIBUTE_MEMORY_TYPE, dp) != CUDA_SUCCESS ||
      mem_type != CU_MEMORYTYPE_DEVICE)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s is not a device pointer", name);
  if (d.ptr_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
      d.ptr_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s: cannot query its allocation", name);
  if (dp + bytes > start + size)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s: %zu bytes needed, its allocation ends %zu bytes after it", name,
                bytes, static_cast<size_t>(start + size - dp));
  return FLUX_ATTN_OK;
}

int check_handle(const flux_attn* h) {
  if (h == nullptr) return fail(FLUX_ATTN_ERR_INVALID_ARG, "handle is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "handle was created on device %d, current device is %d", h->device,
                dev);
  return FLUX_ATTN_OK;
}

int token_count(const flux_attn* h, int txt, int ih, int iw, int rh, int rw, int* n_out) {
  if (txt < 0 || ih < 0 || iw < 0 || rh < 0 || rw < 0)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "negative geometry (txt=%d img=%dx%d ref=%dx%d)", txt, ih, iw, rh, rw);
  const long long n = static_cast<long long>(txt) + static_cast<long long>(ih) * iw +
                      static_cast<long long>(rh) * rw;
  if (n > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "N = %lld tokens exceeds max_tokens = %d", n, h->cfg.max_tokens);
  *n_out = static_cast<int>(n);
  return FLUX_ATTN_OK;
}

size_t row_bytes(const flux_attn* h, int n) {
  return static_cast<size_t>(h->cfg.batch) * n * h->cfg.num_heads * flux::kHeadDim * 2;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, const void* base,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box, const char* what,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const Driver& d = driver();
  if (d.encode == nullptr) return fail(FLUX_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = d.encode(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FLUX_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return FLUX_ATTN_OK;
}

int launch_prologue(flux_attn* h, const void* q, const void* k, int txt, int ih, int iw, int rh, int rw,
                    const int32_t* pos, const float* wq, const float* wk, __nv_bfloat16* qn, __nv_bfloat16* kn,
                    int n, cudaStream_t stream) {
  (void)rh;
  NvtxRange range("flux_attn/qk_norm_rope");
  flux::TokenGeometry geo{pos, txt, ih * iw, iw, rw};
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  const int W = flux::stream_warps<flux::Bf16Rows>(H);
  const long long units = (static_cast<long long>(B) * n + W - 1) / W;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(units, h->num_sms));
  const size_t smem = flux::stream_smem<flux::Bf16Rows>(H);
  flux::StreamArgs a{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), wq, wk,
                     geo, B, n, H, h->cfg.rms_eps, h->rope_tab, h->err};
  a.rot = h->rot;
  flux::qk_norm_rope_kernel<flux::Bf16Rows><<<grid, 32 * W, smem, stream>>>(a, flux::Bf16Rows{qn, kn});
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prologue launch");
  return FLUX_ATTN_OK;
}

size_t pad16(int n) { return (static_cast<size_t>(n) + 15) & ~size_t(15); }

// Key tokens a head repairs for n tokens (VC-Attention): ceil(rho n) in
// [0, n], rho the handle's repair budget.
int repair_count(const flux_attn* h, int n) {
  const double r = std::ceil(static_cast<double>(h->cfg.vc_repair_budget) * static_cast<double>(n));
  if (!(r > 0.0)) return 0;
  return r > n ? n : static_cast<int>(r);
}

// The FP8 prologue: amax of V, Q', K' (after zeroing it), then the codes of
// V transposed, then the E4M3 codes of Q', K' and the scales (last, so that
// the kernel before the attention is the one-wave stream kernel that lets it
// start early).
// V bf16 [B, n, H, 128] in TMA tiles of 64 tokens x 128 dims of one head (for
// its amax and codes), and V^T E4M3 [B*H, 128, pad16(n)] out in tiles of 64 keys.
int encode_v_maps(flux_attn* h, const void* v, void* v8t, int n, CUtensorMap* tv, CUtensorMap* tvt) {
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(flux::kHeadDim), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {flux::kHeadDim * 2ull, static_cast<cuuint64_t>(H) * flux::kHeadDim * 2ull,
                                   static_cast<cuuint64_t>(n) * H * flux::kHeadDim * 2ull};
    const cuuint32_t box[4] = {flux::kHeadDim, 1, flux::kVtTokens, 1};
    int rc = encode_tiled(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dims, strides, box, "V (tiles)",
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  const cuuint64_t np = pad16(n);
  const cuuint64_t dims[3] = {np, static_cast<cuuint64_t>(flux::kHeadDim), static_cast<cuuint64_t>(B) * H};
  const cuuint64_t strides[2] = {np, np * flux::kHeadDim};
  const cuuint32_t box[3] = {flux::kVtTokens, flux::kHeadDim, 1};
  return encode_tiled(tvt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, v8t, dims, strides, box, "V^T (tiles)",
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

// With VC-Attention (repair count R > 0) the quantisers also write the
// per-token K' and V errors, and two more kernels select the repaired tokens
// (sel) and move them out of the codes, writing their exact rows (krep, vrep).
int launch_prologue_fp8(flux_attn* h, const void* q, const void* k, const void* v, int txt, int ih, int iw,
                        int rw, const int32_t* pos, const float* wq, const float* wk, int n, uint8_t* q8,
                        uint8_t* k8, uint8_t* v8t, float* scales, int32_t* sel, __nv_bfloat16* krep,
                        __nv_bfloat16* vrep, cudaStream_t stream) {
  NvtxRange range("flux_attn/fp8_prologue");
  flux::TokenGeometry geo{pos, txt, ih * iw, iw, rw};
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  const size_t amax_bytes = static_cast<size_t>(B) * H * 3 * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(h->amax, 0, amax_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing amax");
  CUtensorMap tv, tvt;
  int rc0 = encode_v_maps(h, v, v8t, n, &tv, &tvt);
  if (rc0) return rc0;
  const dim3 vgrid((n + flux::kVtTokens - 1) / flux::kVtTokens, B * H);
  flux::fp8_vamax_kernel<<<vgrid, flux::kVtThreads, 0, stream>>>(tv, H, h->amax, h->err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "V amax launch");
  // Q', K': the prologue's stream kernel, once reducing to amax, once writing codes
  flux::StreamArgs a{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), wq, wk,
                     geo, B, n, H, h->cfg.rms_eps, h->rope_tab, h->err};
  a.rot = h->rot;
  const long long tokens = static_cast<long long>(B) * n;
  {
    const int W = flux::stream_warps<flux::AmaxRows>(H);
    const unsigned grid = static_cast<unsigned>(std::min<long long>((tokens + W - 1) / W, h->num_sms));
    flux::AmaxRows am{};
    am.amax = h->amax;
    flux::qk_norm_rope_kernel<flux::AmaxRows><<<grid, 32 * W, flux::stream_smem<flux::AmaxRows>(H), stream>>>(a, am);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "amax launch");
  const int R = repair_count(h, n);
  // V^T in the key order of the attention's P.V MMA
  flux::fp8_vt_kernel<true><<<vgrid, flux::kVtThreads, 0, stream>>>(tv, tvt, H, h->amax, h->err,
                                                                   R > 0 ? h->errv : nullptr, n);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "V^T launch");
  {
    const int W = flux::stream_warps<flux::E4m3Rows>(H);
    const unsigned grid = static_cast<unsigned>(std::min<long long>((tokens + W - 1) / W, h->num_sms));
    const flux::E4m3Rows codes{q8, k8, h->amax, scales, H, B * H * 3, R > 0 ? h->errk : nullptr};
    flux::qk_norm_rope_kernel<flux::E4m3Rows>
        <<<grid, 32 * W, flux::stream_smem<flux::E4m3Rows>(H), stream>>>(a, codes);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "quantise launch");
  if (R == 0) return FLUX_ATTN_OK;
  {
    NvtxRange vc_range("flux_attn/vc_repair");
    const size_t sel_smem = n <= flux::vc::kSelectSmemKeys ? static_cast<size_t>(n) * sizeof(uint32_t) : 0;
    flux::vc::vc_select_kernel<<<B * H, flux::vc::kSelectThreads, sel_smem, stream>>>(h->errk, h->errv, n, R, sel);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "repair selection launch");
    const flux::vc::RepairArgs ra{static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), wk,
                                  geo, h->rope_tab, h->rot, n, H, R, h->cfg.rms_eps, scales, sel, k8, v8t,
                                  pad16(n), krep, vrep};
    flux::vc::vc_repair_kernel<<<B * H, flux::vc::kRepairThreads, 0, stream>>>(ra);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "repair launch");
  }
  return FLUX_ATTN_OK;
}

// The attention kernel.  BF16: qn, kn bf16 [B*H, n, 128], v bf16 [B, n, H, 128].
// FP8: qn, kn E4M3 [B*H, n, 128], v E4M3 V^T [B*H, 128, pad16(n)], scales [B*H, 3].
// VC (FP8, R = repair_count > 0): krep, vrep bf16 [B*H, R, 128], and kn, v
// hold the other N - R keys in their first N - R positions.
// SOL (BF16, sol_list set): the block-sparse instance over the lists of
// sol_list_kernel (nb = ceil(n / 128) entries per list).
int launch_attention(flux_attn* h, bool fp8, const void* qn, const void* kn, const void* v, const float* scales,
                     int n, void* out, cudaStream_t stream, const void* krep = nullptr, const void* vrep = nullptr,
                     const uint16_t* sol_list = nullptr, const int* sol_count = nullptr) {
  NvtxRange range(fp8 ? "flux_attn/attention_fp8" : "flux_attn/attention");
  using namespace flux::attn;
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  const size_t esz = fp8 ? 1 : 2;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(n),
                                static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[2] = {HD * esz, static_cast<cuuint64_t>(n) * HD * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), BM, 1};  // one 128-byte swizzle row
    int rc = encode_tiled(&tq, dt, 3, qn, dims, strides, box, "Q'");
    if (rc) return rc;
    rc = encode_tiled(&tk, dt, 3, kn, dims, strides, box, "K'");
    if (rc) return rc;
  }
  if (fp8) {
    const cuuint64_t np = pad16(n);
    const cuuint64_t dims[3] = {np, static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[2] = {np, np * HD};
    const cuuint32_t box[3] = {BN, HD, 1};
    int rc = encode_tiled(&tv, dt, 3, v, dims, strides, box, "V^T");
    if (rc) return rc;
  } else {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {HD * 2ull, static_cast<cuuint64_t>(H) * HD * 2ull,
                                   static_cast<cuuint64_t>(n) * H * HD * 2ull};
    const cuuint32_t box[4] = {64, 1, BN, 1};
    int rc = encode_tiled(&tv, dt, 4, v, dims, strides, box, "V");
    if (rc) return rc;
  }
  CUtensorMap to;
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {HD * 2ull, static_cast<cuuint64_t>(H) * HD * 2ull,
                                   static_cast<cuuint64_t>(n) * H * HD * 2ull};
    const cuuint32_t box[4] = {64, 1, BM, 1};
    int rc = encode_tiled(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, box, "out");
    if (rc) return rc;
  }
  const int R = fp8 ? repair_count(h, n) : 0;
  CUtensorMap tkr = tq, tvr = tq;  // read only by the repair instance
  if (R > 0) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(R),
                                static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[2] = {HD * 2ull, static_cast<cuuint64_t>(R) * HD * 2ull};
    const cuuint32_t box[3] = {64, BN, 1};  // rows >= R arrive as zeros
    int rc = encode_tiled(&tkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, krep, dims, strides, box, "K_rep");
    if (rc) return rc;
    rc = encode_tiled(&tvr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, vrep, dims, strides, box, "V_rep");
    if (rc) return rc;
  }
  Params prm;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.err = h->err;
  prm.scales = scales;
  prm.N = n;
  prm.H = H;
  prm.nrep = (R + BN - 1) / BN;
  prm.rep_keys = R;
  prm.main_keys = n - R;
  prm.nkv = prm.nrep + (n - R + BN - 1) / BN;
  prm.sol_list = sol_list;
  prm.sol_count = sol_count;
  prm.sol_nb = (n + BN - 1) / BN;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  prm.debug = h->cfg.debug_flags;
  // Programmatic stream serialisation: the grid may start before the kernel
  // ahead of it in the stream completes; attn_kernel waits for it
  // (griddepcontrol.wait) before its first global read.
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((n + CTA_ROWS - 1) / CTA_ROWS, B * H);
  lc.blockDim = dim3(R > 0   ? Roles<true, true, false>::THREADS
                     : fp8   ? Roles<true, false, false>::THREADS
                     : sol_list != nullptr ? Roles<false, false, true>::THREADS
                                           : Roles<false, false, false>::THREADS);
  lc.dynamicSmemBytes = fp8 ? smem_bytes<true>() : smem_bytes<false>();
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = R > 0 ? cudaLaunchKernelEx(&lc, attn_kernel<true, true>, tq, tk, tv, to, tkr, tvr, prm)
                  : fp8   ? cudaLaunchKernelEx(&lc, attn_kernel<true, false>, tq, tk, tv, to, tkr, tvr, prm)
                  : sol_list != nullptr
                      ? cudaLaunchKernelEx(&lc, attn_kernel<false, false, true>, tq, tk, tv, to, tkr, tvr, prm)
                      : cudaLaunchKernelEx(&lc, attn_kernel<false, false>, tq, tk, tv, to, tkr, tvr, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return FLUX_ATTN_OK;
}

// Sol-Attention, BF16 Q', K' bf16 [B*H, n, 128]: block means and the keep
// mask (keep: [B*H][nb][nb] uint8).
int launch_sol_mask(flux_attn* h, const void* qn, const void* kn, int n, uint8_t* keep, cudaStream_t stream) {
  NvtxRange range("flux_attn/sol_mask");
  const int BH = h->cfg.batch * h->cfg.num_heads;
  const int nb = (n + flux::sol::kBlock - 1) / flux::sol::kBlock;
  flux::sol::sol_pool_kernel<<<dim3(nb, BH), flux::sol::kPoolThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(qn), static_cast<const __nv_bfloat16*>(kn), n, h->qbar, h->kbar);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "block pooling launch");
  flux::sol::sol_keep_kernel<<<dim3(nb, BH), flux::sol::kThreads, 0, stream>>>(h->qbar, h->kbar, n, h->cfg.sol_tau,
                                                                               keep);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "block mask launch");
  return FLUX_ATTN_OK;
}

// Sol-Attention: the per-CTA key-block lists of a mask, then the sparse attention.
int launch_sol_attention(flux_attn* h, const void* qn, const void* kn, const void* v, const uint8_t* keep, int n,
                         void* out, cudaStream_t stream) {
  const int BH = h->cfg.batch * h->cfg.num_heads;
  const int nb = (n + flux::sol::kBlock - 1) / flux::sol::kBlock;
  const int ncta = (n + flux::attn::CTA_ROWS - 1) / flux::attn::CTA_ROWS;
  flux::sol::sol_list_kernel<<<dim3(ncta, BH), flux::sol::kThreads, 0, stream>>>(keep, nb, h->sol_list,
                                                                                h->sol_count);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "block list launch");
  return launch_attention(h, false, qn, kn, v, nullptr, n, out, stream, nullptr, nullptr, h->sol_list, h->sol_count);
}

// The QKV projection with its fused epilogue: the (cos, sin) table of the
// call's tokens, then the persistent GEMM.
// amax: FP8, the per-(b, h) maxima of the written Q', K', V ([B*H][3], zero on entry); nullptr for BF16.
int launch_qkv(flux_attn* h, const void* x, const void* w, const float* bias, int d_model, int txt, int ih, int iw,
               int rw, const int32_t* pos, const float* wq, const float* wk, void* qn, void* kn, void* v, int n,
               cudaStream_t stream, uint32_t* amax = nullptr) {
  NvtxRange range("flux_attn/qkv_gemm");
  using namespace flux::qkv;
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  const int M = B * n;
  const int F = 3 * H * flux::kHeadDim;
  flux::TokenGeometry geo{pos, txt, ih * iw, iw, rw};
  const int pairs = n * (flux::kHeadDim / 2);
  const int tblocks = std::min((pairs + kTableThreads - 1) / kTableThreads, kTableBlocksPerSm * h->num_sms);
  flux::qkv::rope_table_kernel<<<tblocks, kTableThreads, 0, stream>>>(geo, n, h->rope_tab, h->rot, h->rope);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  CUtensorMap ta, tb;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_model), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_model) * 2};
    const cuuint32_t box[2] = {BK, BM};
    int rc = encode_tiled(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box, "x");
    if (rc) return rc;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_model), static_cast<cuuint64_t>(F)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_model) * 2};
    const cuuint32_t box[2] = {BK, BN};
    int rc = encode_tiled(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dims, strides, box, "w_qkv");
    if (rc) return rc;
  }
  Params p;
  p.bias = bias;
  p.wq = wq;
  p.wk = wk;
  p.rope = h->rope;
  p.qn = static_cast<__nv_bfloat16*>(qn);
  p.kn = static_cast<__nv_bfloat16*>(kn);
  p.v = static_cast<__nv_bfloat16*>(v);
  p.err = h->err;
  p.amax = amax;
  p.M = M;
  p.N = n;
  p.H = H;
  p.D = d_model;
  p.m_tiles = (M + BM - 1) / BM;
  p.n_tiles = (F + BN - 1) / BN;
  p.group_m = group_rows(p.m_tiles, d_model);
  p.eps = h->cfg.rms_eps;
  const int tiles = p.m_tiles * p.n_tiles;
  // Programmatic dependent of the table kernel: producer and MMA warps start
  // on x and W (complete before the table kernel began); the epilogue waits.
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(std::min(tiles, h->num_sms));
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = SMEM_BYTES;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, qkv_gemm_kernel, ta, tb, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "QKV GEMM launch");
  return FLUX_ATTN_OK;
}

// Raise the dynamic shared-memory limit of the prologue and of both
// attention kernels (per device).
cudaError_t set_attention_smem_limits() {
  // the stream kernel's rings and per-warp scratch fit kProSmemBytes (prologue_warps)
  cudaError_t e = cudaFuncSetAttribute(flux::qk_norm_rope_kernel<flux::Bf16Rows>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, flux::kProSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::qk_norm_rope_kernel<flux::AmaxRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           flux::kProSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::qk_norm_rope_kernel<flux::E4m3Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           flux::kProSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::vc::vc_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(flux::vc::kSelectSmemKeys * sizeof(uint32_t)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::qkv::qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(flux::qkv::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::attn::attn_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(flux::attn::smem_bytes<false>()));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::attn::attn_kernel<false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(flux::attn::smem_bytes<false>()));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flux::attn::attn_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(flux::attn::smem_bytes<true>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(flux::attn::attn_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(flux::attn::smem_bytes<true>()));
}

}  // namespace

extern "C" {

const char* flux_attn_status_string(int status) {
  switch (status) {
    case FLUX_ATTN_OK: return "ok";
    case FLUX_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case FLUX_ATTN_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case FLUX_ATTN_ERR_OOM: return "out of device memory";
    case FLUX_ATTN_ERR_CUDA: return "CUDA error";
    case FLUX_ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* flux_attn_last_error(void) { return g_last_error.c_str(); }

int flux_attn_create(const flux_attn_config* cfg, flux_attn_t* out) {
  g_last_error.clear();
  if (out == nullptr) return fail(FLUX_ATTN_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (cfg == nullptr) return fail(FLUX_ATTN_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->head_dim != flux::kHeadDim)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "head_dim = %d, only 128 is built", cfg->head_dim);
  if (cfg->batch < 1 || cfg->num_heads < 1 || cfg->max_tokens < 1)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "batch, num_heads and max_tokens must be >= 1");
  if (static_cast<long long>(cfg->batch) * cfg->num_heads > 65535)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "batch * num_heads must be <= 65535");
  if (cfg->num_heads > flux::kProMaxHeads)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "num_heads = %d, at most %d are built", cfg->num_heads, flux::kProMaxHeads);
  if (cfg->max_tokens > (1 << 24)) return fail(FLUX_ATTN_ERR_INVALID_ARG, "max_tokens must be <= 2^24");
  const int* ax = cfg->axes_dim;
  if (ax[0] < 0 || ax[1] < 0 || ax[2] < 0 || (ax[0] | ax[1] | ax[2]) & 1 ||
      ax[0] + ax[1] + ax[2] != cfg->head_dim)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "axes_dim (%d, %d, %d) must be even and sum to head_dim", ax[0], ax[1],
                ax[2]);
  // The prologue gives each lane 8 consecutive dims; they must stay in one axis block.
  if (ax[0] % 8 || ax[1] % 8)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "axes_dim[0] and axes_dim[1] must be multiples of 8");
  if (!(cfg->rope_theta > 0.f) || !(cfg->rms_eps >= 0.f))
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");
  if (cfg->precision != FLUX_ATTN_BF16 && cfg->precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "unknown precision %d", cfg->precision);
  if (!(cfg->vc_repair_budget >= 0.f && cfg->vc_repair_budget <= 1.f))
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "vc_repair_budget must be in [0, 1]");
  if (cfg->vc_repair_budget > 0.f && cfg->precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "vc_repair_budget > 0 needs precision FLUX_ATTN_FP8_E4M3");
  if (!(cfg->sol_tau >= 0.f) || cfg->sol_tau > 3.0e38f)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "sol_tau must be finite and >= 0");
  if (cfg->sol_tau > 0.f && cfg->precision != FLUX_ATTN_BF16)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "sol_tau > 0 needs precision FLUX_ATTN_BF16");
  if (cfg->sol_tau > 0.f && cfg->max_tokens > kSolMaxTokens)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "Sol-Attention is built for max_tokens <= %d", kSolMaxTokens);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d, this library is built for sm_103a", dev,
                prop.major, prop.minor);
  if (driver().encode == nullptr || driver().ptr_attr == nullptr)
    return fail(FLUX_ATTN_ERR_CUDA, "driver entry points unavailable");
  e = set_attention_smem_limits();
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");

  flux_attn* h = new flux_attn();
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  // RoPE table: pair j of axis block a (local index jj) turns by pos_a * theta^(-2 jj / d_a).
  {
    int j = 0;
    for (int a = 0; a < 3; ++a)
      for (int jj = 0; jj < ax[a] / 2; ++jj, ++j) {
        h->rope_tab.freq[j] = static_cast<float>(std::pow(static_cast<double>(cfg->rope_theta), -2.0 * jj / ax[a]));
        h->rope_tab.axis[j] = a;
      }
  }
  // Workspace, each piece 256-byte aligned:
  //   both  Q', K' bf16 [B, H, max_tokens, 128], V bf16 [B, max_tokens, H, 128] and the
  //         (cos, sin) table of the QKV projection (FP8: its bf16 outputs before the codes)
  //   FP8   Q', K' E4M3 [B, H, max_tokens, 128], V^T E4M3 [B, H, 128, pad16(max_tokens)],
  //         amax and scales [B, H, 3]
  //   VC / SOL  their buffers (below); the per-position rotation table; the device error word
  const size_t bh = static_cast<size_t>(cfg->batch) * cfg->num_heads;
  const bool fp8 = cfg->precision == FLUX_ATTN_FP8_E4M3;
  const auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t qk_bytes = al(bh * cfg->max_tokens * flux::kHeadDim * 2);
  const size_t q8_bytes = fp8 ? al(bh * cfg->max_tokens * flux::kHeadDim) : 0;
  const size_t vt_bytes = fp8 ? al(bh * flux::kHeadDim * pad16(cfg->max_tokens)) : 0;
  const size_t sc_bytes = fp8 ? al(bh * 3 * sizeof(float)) : 0;
  const size_t rope_bytes = al(static_cast<size_t>(cfg->max_tokens) * (flux::kHeadDim / 2) * sizeof(float2));
  const size_t rot_bytes = al(static_cast<size_t>(flux::kRotPositions) * (flux::kHeadDim / 2) * sizeof(float2));
  const size_t v_bytes = qk_bytes;
  h->r_max = repair_count(h, cfg->max_tokens);
  const size_t vc_err_bytes = h->r_max > 0 ? al(bh * cfg->max_tokens * sizeof(float)) : 0;
  const size_t vc_sel_bytes = h->r_max > 0 ? al(bh * h->r_max * sizeof(int32_t)) : 0;
  const size_t vc_row_bytes = h->r_max > 0 ? al(bh * h->r_max * flux::kHeadDim * 2) : 0;
  const size_t f8_off = 2 * qk_bytes + rope_bytes + v_bytes;
  const size_t vc_off = f8_off + 2 * q8_bytes + vt_bytes + 2 * sc_bytes;
  const bool sol = cfg->sol_tau > 0.f;
  const size_t nb_max = (static_cast<size_t>(cfg->max_tokens) + 127) / 128;
  const size_t ncta_max = (static_cast<size_t>(cfg->max_tokens) + 255) / 256;
  const size_t sol_bar_bytes = sol ? al(bh * nb_max * flux::kHeadDim * sizeof(float)) : 0;
  const size_t sol_keep_bytes = sol ? al(bh * nb_max * nb_max) : 0;
  const size_t sol_list_bytes = sol ? al(bh * ncta_max * nb_max * sizeof(uint16_t)) : 0;
  const size_t sol_count_bytes = sol ? al(bh * ncta_max * sizeof(int)) : 0;
  const size_t sol_off = vc_off + 2 * vc_err_bytes + vc_sel_bytes + 2 * vc_row_bytes;
  const size_t rot_off = sol_off + 2 * sol_bar_bytes + sol_keep_bytes + sol_list_bytes + sol_count_bytes;
  const size_t err_off = rot_off + rot_bytes;
  h->ws_bytes = err_off + 256;
  e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) {
    const size_t want = h->ws_bytes;
    delete h;
    cudaGetLastError();
    return fail(FLUX_ATTN_ERR_OOM, "cudaMalloc(%zu) failed: %s", want, cudaGetErrorString(e));
  }
  uint8_t* base = static_cast<uint8_t*>(h->ws);
  h->qn = reinterpret_cast<__nv_bfloat16*>(base);
  h->kn = reinterpret_cast<__nv_bfloat16*>(base + qk_bytes);
  h->rope = reinterpret_cast<float2*>(base + 2 * qk_bytes);
  h->vw = reinterpret_cast<__nv_bfloat16*>(base + 2 * qk_bytes + rope_bytes);
  if (fp8) {
    h->q8 = base + f8_off;
    h->k8 = base + f8_off + q8_bytes;
    h->v8t = base + f8_off + 2 * q8_bytes;
    h->amax = reinterpret_cast<uint32_t*>(base + f8_off + 2 * q8_bytes + vt_bytes);
    h->scales = reinterpret_cast<float*>(base + f8_off + 2 * q8_bytes + vt_bytes + sc_bytes);
  }
  if (h->r_max > 0) {
    h->errk = reinterpret_cast<float*>(base + vc_off);
    h->errv = reinterpret_cast<float*>(base + vc_off + vc_err_bytes);
    h->sel = reinterpret_cast<int32_t*>(base + vc_off + 2 * vc_err_bytes);
    h->krep = reinterpret_cast<__nv_bfloat16*>(base + vc_off + 2 * vc_err_bytes + vc_sel_bytes);
    h->vrep = reinterpret_cast<__nv_bfloat16*>(base + vc_off + 2 * vc_err_bytes + vc_sel_bytes + vc_row_bytes);
  }
  if (sol) {
    h->qbar = reinterpret_cast<float*>(base + sol_off);
    h->kbar = reinterpret_cast<float*>(base + sol_off + sol_bar_bytes);
    h->keep = base + sol_off + 2 * sol_bar_bytes;
    h->sol_list = reinterpret_cast<uint16_t*>(base + sol_off + 2 * sol_bar_bytes + sol_keep_bytes);
    h->sol_count = reinterpret_cast<int*>(base + sol_off + 2 * sol_bar_bytes + sol_keep_bytes + sol_list_bytes);
  }
  h->err = reinterpret_cast<uint32_t*>(base + err_off);
  h->rot = reinterpret_cast<float2*>(base + rot_off);
  e = cudaMemset(h->err, 0, 256);
  if (e == cudaSuccess) {
    // the rotation table, once (the handle's calls may come on any stream)
    constexpr int kRotElems = flux::kRotPositions * (flux::kHeadDim / 2);
    flux::rot_table_kernel<<<(kRotElems + 255) / 256, 256>>>(h->rope_tab, h->rot);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return cuda_fail(e, "initialising the workspace");
  }
  *out = h;
  return FLUX_ATTN_OK;
}

int flux_attn_destroy(flux_attn_t h) {
  if (h == nullptr) return FLUX_ATTN_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != h->device) cudaSetDevice(h->device);
  cudaError_t e = cudaFree(h->ws);
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree");
  return FLUX_ATTN_OK;
}

size_t flux_attn_workspace_bytes(flux_attn_t h) { return h ? h->ws_bytes : 0; }

int flux_attn_launches_per_forward(flux_attn_t h, int n_tokens) {
  if (h == nullptr || n_tokens <= 0) return 0;
  // BF16: prologue + attention; FP8: V amax + Q'/K' amax + Q'/K' codes +
  // V^T codes + attention (the amax zeroing is a cudaMemsetAsync, not a
  // kernel of this library).
  // VC-Attention adds the repair selection and the repair kernel.
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3) return 2;
  return repair_count(h, n_tokens) > 0 ? 7 : 5;
}

static int check_common(flux_attn* h, const void* q, const void* k, int txt, int ih, int iw, int rh, int rw,
                        const int32_t* pos, const float* wq, const float* wk, int* n) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = token_count(h, txt, ih, iw, rh, rw, n);
  if (rc) return rc;
  if (*n == 0) return FLUX_ATTN_OK;
  const size_t bytes = row_bytes(h, *n);
  if ((rc = check_buffer(q, bytes, "q"))) return rc;
  if ((rc = check_buffer(k, bytes, "k"))) return rc;
  if ((rc = check_buffer(wq, flux::kHeadDim * sizeof(float), "q_norm_w"))) return rc;
  if ((rc = check_buffer(wk, flux::kHeadDim * sizeof(float), "k_norm_w"))) return rc;
  if (pos != nullptr && (rc = check_buffer(pos, static_cast<size_t>(*n) * 3 * sizeof(int32_t), "pos_ids")))
    return rc;
  return FLUX_ATTN_OK;
}

int flux_attn_prologue(flux_attn_t h, const void* q, const void* k, int txt_len, int img_h, int img_w, int ref_h,
                       int ref_w, const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w, void* qn,
                       void* kn, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_prologue");
  int n = 0;
  int rc = check_common(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n);
  if (rc || n == 0) return rc;
  if (h->cfg.precision != FLUX_ATTN_BF16)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_prologue needs a BF16 handle");
  const size_t bytes = row_bytes(h, n);
  if ((rc = check_buffer(qn, bytes, "qn"))) return rc;
  if ((rc = check_buffer(kn, bytes, "kn"))) return rc;
  return launch_prologue(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                         static_cast<__nv_bfloat16*>(qn), static_cast<__nv_bfloat16*>(kn), n, stream);
}

int flux_attn_attend(flux_attn_t h, const void* qn, const void* kn, const void* v, int n_tokens, void* out,
                     cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_attend");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_BF16)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_attend needs a BF16 handle");
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "n_tokens = %d outside [0, max_tokens = %d]", n_tokens,
                h->cfg.max_tokens);
  if (n_tokens == 0) return FLUX_ATTN_OK;
  const size_t bytes = row_bytes(h, n_tokens);
  if ((rc = check_buffer(qn, bytes, "qn"))) return rc;
  if ((rc = check_buffer(kn, bytes, "kn"))) return rc;
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if ((rc = check_buffer(out, bytes, "out"))) return rc;
  return launch_attention(h, false, qn, kn, v, nullptr, n_tokens, out, stream);
}

int flux_attn_forward(flux_attn_t h, const void* q, const void* k, const void* v, int txt_len, int img_h,
                      int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                      const float* k_norm_w, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_forward");
  int n = 0;
  int rc = check_common(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n);
  if (rc || n == 0) return rc;
  const size_t bytes = row_bytes(h, n);
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if ((rc = check_buffer(out, bytes, "out"))) return rc;
  if (out == q || out == k || out == v) return fail(FLUX_ATTN_ERR_INVALID_ARG, "out aliases an input");
  if (h->cfg.precision == FLUX_ATTN_BF16) {
    rc = launch_prologue(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, h->qn, h->kn,
                         n, stream);
    if (rc) return rc;
    return launch_attention(h, false, h->qn, h->kn, v, nullptr, n, out, stream);
  }
  rc = launch_prologue_fp8(h, q, k, v, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, n, h->q8, h->k8,
                           h->v8t, h->scales, h->sel, h->krep, h->vrep, stream);
  if (rc) return rc;
  return launch_attention(h, true, h->q8, h->k8, h->v8t, h->scales, n, out, stream, h->krep, h->vrep);
}

int flux_attn_prologue_fp8(flux_attn_t h, const void* q, const void* k, const void* v, int txt_len, int img_h,
                           int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                           const float* k_norm_w, void* q8, void* k8, void* v8t, float* scales,
                           cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_prologue_fp8");
  int n = 0;
  int rc = check_common(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n);
  if (rc || n == 0) return rc;
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_prologue_fp8 needs an FP8 handle");
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  if ((rc = check_buffer(v, row_bytes(h, n), "v"))) return rc;
  if ((rc = check_buffer(q8, bh * n * flux::kHeadDim, "q8"))) return rc;
  if ((rc = check_buffer(k8, bh * n * flux::kHeadDim, "k8"))) return rc;
  if ((rc = check_buffer(v8t, bh * flux::kHeadDim * pad16(n), "v8t"))) return rc;
  if ((rc = check_buffer(scales, bh * 3 * sizeof(float), "scales"))) return rc;
  if (repair_count(h, n) > 0)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "a VC-Attention handle takes flux_attn_prologue_fp8_vc");
  return launch_prologue_fp8(h, q, k, v, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, n,
                             static_cast<uint8_t*>(q8), static_cast<uint8_t*>(k8), static_cast<uint8_t*>(v8t),
                             scales, nullptr, nullptr, nullptr, stream);
}

int flux_attn_prologue_fp8_vc(flux_attn_t h, const void* q, const void* k, const void* v, int txt_len, int img_h,
                              int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                              const float* k_norm_w, void* q8, void* k8, void* v8t, float* scales,
                              int32_t* repair_idx, void* k_rep, void* v_rep, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_prologue_fp8_vc");
  int n = 0;
  int rc = check_common(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n);
  if (rc || n == 0) return rc;
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_prologue_fp8_vc needs an FP8 handle");
  const int R = repair_count(h, n);
  if (R == 0) return fail(FLUX_ATTN_ERR_INVALID_ARG, "the handle repairs no token for %d tokens", n);
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  if ((rc = check_buffer(v, row_bytes(h, n), "v"))) return rc;
  if ((rc = check_buffer(q8, bh * n * flux::kHeadDim, "q8"))) return rc;
  if ((rc = check_buffer(k8, bh * n * flux::kHeadDim, "k8"))) return rc;
  if ((rc = check_buffer(v8t, bh * flux::kHeadDim * pad16(n), "v8t"))) return rc;
  if ((rc = check_buffer(scales, bh * 3 * sizeof(float), "scales"))) return rc;
  if ((rc = check_buffer(repair_idx, bh * R * sizeof(int32_t), "repair_idx"))) return rc;
  if ((rc = check_buffer(k_rep, bh * R * flux::kHeadDim * 2, "k_rep"))) return rc;
  if ((rc = check_buffer(v_rep, bh * R * flux::kHeadDim * 2, "v_rep"))) return rc;
  return launch_prologue_fp8(h, q, k, v, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, n,
                             static_cast<uint8_t*>(q8), static_cast<uint8_t*>(k8), static_cast<uint8_t*>(v8t),
                             scales, repair_idx, static_cast<__nv_bfloat16*>(k_rep),
                             static_cast<__nv_bfloat16*>(v_rep), stream);
}

int flux_attn_vc_repair_count(flux_attn_t h, int n_tokens) {
  if (h == nullptr || n_tokens <= 0 || h->cfg.precision != FLUX_ATTN_FP8_E4M3) return 0;
  return repair_count(h, n_tokens);
}

int flux_attn_attend_fp8(flux_attn_t h, const void* q8, const void* k8, const void* v8t, const float* scales,
                         int n_tokens, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_attend_fp8");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_attend_fp8 needs an FP8 handle");
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "n_tokens = %d outside [0, max_tokens = %d]", n_tokens,
                h->cfg.max_tokens);
  if (n_tokens == 0) return FLUX_ATTN_OK;
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  if ((rc = check_buffer(q8, bh * n_tokens * flux::kHeadDim, "q8"))) return rc;
  if ((rc = check_buffer(k8, bh * n_tokens * flux::kHeadDim, "k8"))) return rc;
  if ((rc = check_buffer(v8t, bh * flux::kHeadDim * pad16(n_tokens), "v8t"))) return rc;
  if ((rc = check_buffer(scales, bh * 3 * sizeof(float), "scales"))) return rc;
  if ((rc = check_buffer(out, row_bytes(h, n_tokens), "out"))) return rc;
  if (repair_count(h, n_tokens) > 0)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "a VC-Attention handle takes flux_attn_attend_fp8_vc");
  return launch_attention(h, true, q8, k8, v8t, scales, n_tokens, out, stream);
}

int flux_attn_attend_fp8_vc(flux_attn_t h, const void* q8, const void* k8, const void* v8t, const float* scales,
                            const void* k_rep, const void* v_rep, int n_tokens, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_attend_fp8_vc");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_attend_fp8_vc needs an FP8 handle");
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "n_tokens = %d outside [0, max_tokens = %d]", n_tokens,
                h->cfg.max_tokens);
  if (n_tokens == 0) return FLUX_ATTN_OK;
  const int R = repair_count(h, n_tokens);
  if (R == 0) return fail(FLUX_ATTN_ERR_INVALID_ARG, "the handle repairs no token for %d tokens", n_tokens);
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  if ((rc = check_buffer(q8, bh * n_tokens * flux::kHeadDim, "q8"))) return rc;
  if ((rc = check_buffer(k8, bh * n_tokens * flux::kHeadDim, "k8"))) return rc;
  if ((rc = check_buffer(v8t, bh * flux::kHeadDim * pad16(n_tokens), "v8t"))) return rc;
  if ((rc = check_buffer(scales, bh * 3 * sizeof(float), "scales"))) return rc;
  if ((rc = check_buffer(k_rep, bh * R * flux::kHeadDim * 2, "k_rep"))) return rc;
  if ((rc = check_buffer(v_rep, bh * R * flux::kHeadDim * 2, "v_rep"))) return rc;
  if ((rc = check_buffer(out, row_bytes(h, n_tokens), "out"))) return rc;
  return launch_attention(h, true, q8, k8, v8t, scales, n_tokens, out, stream, k_rep, v_rep);
}

static int sol_handle(flux_attn* h, const char* what) {
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_BF16 || !(h->cfg.sol_tau > 0.f))
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "%s needs a BF16 handle with sol_tau > 0", what);
  return FLUX_ATTN_OK;
}

int flux_attn_sol_mask(flux_attn_t h, const void* qn, const void* kn, int n_tokens, uint8_t* keep,
                       cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_sol_mask");
  int rc = sol_handle(h, "flux_attn_sol_mask");
  if (rc) return rc;
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "n_tokens = %d outside [0, max_tokens = %d]", n_tokens,
                h->cfg.max_tokens);
  if (n_tokens == 0) return FLUX_ATTN_OK;
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  const size_t nb = (static_cast<size_t>(n_tokens) + 127) / 128;
  if ((rc = check_buffer(qn, row_bytes(h, n_tokens), "qn"))) return rc;
  if ((rc = check_buffer(kn, row_bytes(h, n_tokens), "kn"))) return rc;
  if ((rc = check_buffer(keep, bh * nb * nb, "keep"))) return rc;
  return launch_sol_mask(h, qn, kn, n_tokens, keep, stream);
}

int flux_attn_attend_sol(flux_attn_t h, const void* qn, const void* kn, const void* v, const uint8_t* keep,
                         int n_tokens, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_attend_sol");
  int rc = sol_handle(h, "flux_attn_attend_sol");
  if (rc) return rc;
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "n_tokens = %d outside [0, max_tokens = %d]", n_tokens,
                h->cfg.max_tokens);
  if (n_tokens == 0) return FLUX_ATTN_OK;
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  const size_t nb = (static_cast<size_t>(n_tokens) + 127) / 128;
  const size_t bytes = row_bytes(h, n_tokens);
  if ((rc = check_buffer(qn, bytes, "qn"))) return rc;
  if ((rc = check_buffer(kn, bytes, "kn"))) return rc;
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if ((rc = check_buffer(keep, bh * nb * nb, "keep"))) return rc;
  if ((rc = check_buffer(out, bytes, "out"))) return rc;
  return launch_sol_attention(h, qn, kn, v, keep, n_tokens, out, stream);
}

int flux_attn_forward_sol(flux_attn_t h, const void* q, const void* k, const void* v, int txt_len, int img_h,
                          int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                          const float* k_norm_w, float timestep, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_forward_sol");
  int rc = sol_handle(h, "flux_attn_forward_sol");
  if (rc) return rc;
  int n = 0;
  rc = check_common(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n);
  if (rc || n == 0) return rc;
  const size_t bytes = row_bytes(h, n);
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if ((rc = check_buffer(out, bytes, "out"))) return rc;
  if (out == q || out == k || out == v) return fail(FLUX_ATTN_ERR_INVALID_ARG, "out aliases an input");
  rc = launch_prologue(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, h->qn, h->kn, n,
                       stream);
  if (rc) return rc;
  if (timestep > h->cfg.sol_disabled_until_timestep)  // the early (noisy) steps stay dense
    return launch_attention(h, false, h->qn, h->kn, v, nullptr, n, out, stream);
  rc = launch_sol_mask(h, h->qn, h->kn, n, h->keep, stream);
  if (rc) return rc;
  return launch_sol_attention(h, h->qn, h->kn, v, h->keep, n, out, stream);
}

// Arguments of the QKV projection shared by its BF16 and FP8 entry points.
static int qkv_common(flux_attn* h, const void* x, const void* w_qkv, const float* b_qkv, int d_model, int txt_len,
                      int img_h, int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                      const float* k_norm_w, int* n_out) {
  int rc = 0;
  if (d_model < flux::qkv::BK || d_model % flux::qkv::BK || d_model > (1 << 16))
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "d_model = %d must be a multiple of %d in [%d, 65536]", d_model,
                flux::qkv::BK, flux::qkv::BK);
  int n = 0;
  if ((rc = token_count(h, txt_len, img_h, img_w, ref_h, ref_w, &n))) return rc;
  *n_out = n;
  if (n == 0) return FLUX_ATTN_OK;
  const size_t M = static_cast<size_t>(h->cfg.batch) * n;
  const size_t F = 3ull * h->cfg.num_heads * flux::kHeadDim;
  if ((rc = check_buffer(x, M * d_model * 2, "x"))) return rc;
  if ((rc = check_buffer(w_qkv, F * d_model * 2, "w_qkv"))) return rc;
  if (b_qkv != nullptr && (rc = check_buffer(b_qkv, F * sizeof(float), "b_qkv"))) return rc;
  if ((rc = check_buffer(q_norm_w, flux::kHeadDim * sizeof(float), "q_norm_w"))) return rc;
  if ((rc = check_buffer(k_norm_w, flux::kHeadDim * sizeof(float), "k_norm_w"))) return rc;
  if (pos_ids != nullptr && (rc = check_buffer(pos_ids, static_cast<size_t>(n) * 3 * sizeof(int32_t), "pos_ids")))
    return rc;
  return FLUX_ATTN_OK;
}

// The FP8 QKV projection into q8, k8, v8t, scales: the GEMM writes bf16 Q', K',
// V to the workspace and reduces their per-(b, h) amax, then the codes.
static int launch_qkv_fp8(flux_attn* h, const void* x, const void* w_qkv, const float* b_qkv, int d_model,
                          int txt_len, int img_h, int img_w, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                          const float* k_norm_w, int n, uint8_t* q8, uint8_t* k8, uint8_t* v8t, float* scales,
                          cudaStream_t stream) {
  const int B = h->cfg.batch, H = h->cfg.num_heads;
  cudaError_t e = cudaMemsetAsync(h->amax, 0, static_cast<size_t>(B) * H * 3 * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing amax");
  int rc = launch_qkv(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, h->qn,
                      h->kn, h->vw, n, stream, h->amax);
  if (rc) return rc;
  NvtxRange range("flux_attn/fp8_codes");
  CUtensorMap tv, tvt;
  if ((rc = encode_v_maps(h, h->vw, v8t, n, &tv, &tvt))) return rc;
  const dim3 vgrid((n + flux::kVtTokens - 1) / flux::kVtTokens, B * H);
  // the key order of the attention's P.V MMA
  flux::fp8_vt_kernel<true><<<vgrid, flux::kVtThreads, 0, stream>>>(tv, tvt, H, h->amax, h->err, nullptr, n);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "V^T launch");
  const size_t items = 2ull * B * H * n * flux::kHeadDim / 16;
  const unsigned grid = static_cast<unsigned>(
      std::min<size_t>((items + flux::kCodesThreads - 1) / flux::kCodesThreads, 8ull * h->num_sms));
  flux::fp8_codes_kernel<<<grid, flux::kCodesThreads, 0, stream>>>(h->qn, h->kn, n, B * H, h->amax, q8, k8, scales);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "codes launch");
  return FLUX_ATTN_OK;
}

int flux_attn_qkv_fp8(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv, int d_model, int txt_len,
                      int img_h, int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                      const float* k_norm_w, void* q8, void* k8, void* v8t, float* scales, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_qkv_fp8");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "flux_attn_qkv_fp8 needs an FP8 handle");
  if (h->cfg.vc_repair_budget > 0.f)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "the QKV projection has no VC-Attention repair");
  int n = 0;
  if ((rc = qkv_common(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                       k_norm_w, &n)) || n == 0)
    return rc;
  const size_t bh = static_cast<size_t>(h->cfg.batch) * h->cfg.num_heads;
  if ((rc = check_buffer(q8, bh * n * flux::kHeadDim, "q8"))) return rc;
  if ((rc = check_buffer(k8, bh * n * flux::kHeadDim, "k8"))) return rc;
  if ((rc = check_buffer(v8t, bh * flux::kHeadDim * pad16(n), "v8t"))) return rc;
  if ((rc = check_buffer(scales, bh * 3 * sizeof(float), "scales"))) return rc;
  return launch_qkv_fp8(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, n,
                        static_cast<uint8_t*>(q8), static_cast<uint8_t*>(k8), static_cast<uint8_t*>(v8t), scales,
                        stream);
}

int flux_attn_qkv(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv, int d_model, int txt_len,
                  int img_h, int img_w, int ref_h, int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                  const float* k_norm_w, void* qn, void* kn, void* v, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_qkv");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision != FLUX_ATTN_BF16)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "flux_attn_qkv needs a BF16 handle (FP8: flux_attn_qkv_fp8)");
  if (d_model < flux::qkv::BK || d_model % flux::qkv::BK || d_model > (1 << 16))
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "d_model = %d must be a multiple of %d in [%d, 65536]", d_model,
                flux::qkv::BK, flux::qkv::BK);
  int n = 0;
  if ((rc = token_count(h, txt_len, img_h, img_w, ref_h, ref_w, &n))) return rc;
  if (n == 0) return FLUX_ATTN_OK;
  const size_t M = static_cast<size_t>(h->cfg.batch) * n;
  const size_t F = 3ull * h->cfg.num_heads * flux::kHeadDim;
  if ((rc = check_buffer(x, M * d_model * 2, "x"))) return rc;
  if ((rc = check_buffer(w_qkv, F * d_model * 2, "w_qkv"))) return rc;
  if (b_qkv != nullptr && (rc = check_buffer(b_qkv, F * sizeof(float), "b_qkv"))) return rc;
  if ((rc = check_buffer(q_norm_w, flux::kHeadDim * sizeof(float), "q_norm_w"))) return rc;
  if ((rc = check_buffer(k_norm_w, flux::kHeadDim * sizeof(float), "k_norm_w"))) return rc;
  if (pos_ids != nullptr && (rc = check_buffer(pos_ids, static_cast<size_t>(n) * 3 * sizeof(int32_t), "pos_ids")))
    return rc;
  const size_t bytes = row_bytes(h, n);
  if ((rc = check_buffer(qn, bytes, "qn"))) return rc;
  if ((rc = check_buffer(kn, bytes, "kn"))) return rc;
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if (qn == kn || qn == v || kn == v || qn == x || kn == x || v == x)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "qn, kn, v and x must be distinct buffers");
  return launch_qkv(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, qn, kn,
                    v, n, stream);
}

int flux_attn_forward_hidden(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv, int d_model,
                             int txt_len, int img_h, int img_w, int ref_h, int ref_w, const int32_t* pos_ids,
                             const float* q_norm_w, const float* k_norm_w, void* out, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_forward_hidden");
  int rc = check_handle(h);
  if (rc) return rc;
  if (h->cfg.precision == FLUX_ATTN_FP8_E4M3 && h->cfg.vc_repair_budget > 0.f)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "the QKV projection has no VC-Attention repair");
  int n = 0;
  if ((rc = token_count(h, txt_len, img_h, img_w, ref_h, ref_w, &n))) return rc;
  if (n == 0) return FLUX_ATTN_OK;
  if ((rc = check_buffer(out, row_bytes(h, n), "out"))) return rc;
  if (out == x) return fail(FLUX_ATTN_ERR_INVALID_ARG, "out aliases x");
  if (h->cfg.precision == FLUX_ATTN_FP8_E4M3) {
    if ((rc = qkv_common(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                         k_norm_w, &n)))
      return rc;
    rc = launch_qkv_fp8(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_w, pos_ids, q_norm_w, k_norm_w, n,
                        h->q8, h->k8, h->v8t, h->scales, stream);
    if (rc) return rc;
    return launch_attention(h, true, h->q8, h->k8, h->v8t, h->scales, n, out, stream);
  }
  // the projection's own checks, with the handle's workspace as its outputs
  rc = flux_attn_qkv(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                     h->qn, h->kn, h->vw, stream);
  if (rc) return rc;
  return launch_attention(h, false, h->qn, h->kn, h->vw, nullptr, n, out, stream);
}

int flux_attn_sync_status(flux_attn_t h, cudaStream_t stream) {
  g_last_error.clear();
  int rc = check_handle(h);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word != 0) {
    e = cudaMemset(h->err, 0, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    return fail(FLUX_ATTN_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out (error word 0x%x)", word);
  }
  return FLUX_ATTN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.
//
// Some callers must not allocate device memory on the call path: inference
// engines that reserve and plan all device memory once at start-up and forbid
// any later cudaMalloc, plugin hosts that give a plugin only the buffers it
// declared, and latency-critical callers that cannot take the implicit
// device-wide synchronisation that cudaMalloc / cudaFree may cause.  For them
// flux_attn_forward_noalloc runs the same two kernels as flux_attn_forward
// without a handle: the normalised Q'/K' scratch and the device error word
// live in the file-scope array below, which the CUDA module holds on every
// device that loads this library until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocWordBytes = 256;                       // device error word (+ padding)
constexpr size_t kNoAllocQKBytes = size_t(16) << 20;            // Q' and K', bf16
constexpr size_t kNoAllocRowBytes = flux::kHeadDim * 2;         // one bf16 head row
constexpr long long kNoAllocMaxTokenHeads = kNoAllocQKBytes / (2 * kNoAllocRowBytes);  // 32768

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocWordBytes + kNoAllocQKBytes];

struct NoAllocDevice {
  std::once_flag once;
  int status = FLUX_ATTN_ERR_CUDA;
  uint8_t* base = nullptr;  // device address of g_noalloc_scratch on this device
  std::string msg;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device, with that device current: look up the device address of
// the scratch array (the host-side symbol is only a stand-in) and raise the
// attention kernel's dynamic shared-memory limit.
int noalloc_setup(int dev, uint8_t** base) {
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kNoAllocMaxDevices);
  NoAllocDevice& d = g_noalloc_dev[dev];
  std::call_once(d.once, [&d] {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      d.msg = std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e);
      return;
    }
    e = set_attention_smem_limits();
    if (e != cudaSuccess) {
      d.msg = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return;
    }
    d.base = static_cast<uint8_t*>(p);
    d.status = FLUX_ATTN_OK;
  });
  if (d.status != FLUX_ATTN_OK) return fail(d.status, "%s", d.msg.c_str());
  *base = d.base;
  return FLUX_ATTN_OK;
}

}  // namespace

extern "C" int flux_attn_forward_noalloc(const flux_attn_config* cfg, const void* q, const void* k, const void* v,
                                         int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                                         const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                                         void* out, uint32_t* device_error, cudaStream_t stream) {
  g_last_error.clear();
  NvtxRange range("flux_attn_forward_noalloc");
  if (cfg == nullptr) return fail(FLUX_ATTN_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->head_dim != flux::kHeadDim)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "head_dim = %d, only 128 is built", cfg->head_dim);
  if (cfg->precision != FLUX_ATTN_BF16 && cfg->precision != FLUX_ATTN_FP8_E4M3)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "unknown precision %d", cfg->precision);
  if (cfg->precision != FLUX_ATTN_BF16)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "the allocation-free forward is BF16 only");
  if (cfg->vc_repair_budget != 0.f)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "vc_repair_budget > 0 needs precision FLUX_ATTN_FP8_E4M3");
  if (cfg->sol_tau != 0.f)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "the allocation-free forward is dense only (sol_tau must be 0)");
  if (cfg->batch < 1 || cfg->num_heads < 1 || cfg->max_tokens < 1)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "batch, num_heads and max_tokens must be >= 1");
  if (cfg->num_heads > flux::kProMaxHeads)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "num_heads = %d, at most %d are built", cfg->num_heads, flux::kProMaxHeads);
  const int* ax = cfg->axes_dim;
  if (ax[0] < 0 || ax[1] < 0 || ax[2] < 0 || (ax[0] | ax[1] | ax[2]) & 1 ||
      ax[0] + ax[1] + ax[2] != cfg->head_dim)
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "axes_dim (%d, %d, %d) must be even and sum to head_dim", ax[0], ax[1],
                ax[2]);
  if (ax[0] % 8 || ax[1] % 8)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "axes_dim[0] and axes_dim[1] must be multiples of 8");
  if (!(cfg->rope_theta > 0.f) || !(cfg->rms_eps >= 0.f))
    return fail(FLUX_ATTN_ERR_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(FLUX_ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d, this library is built for sm_103a", dev, major,
                minor);

  // A handle-shaped view of this call; nothing in it is allocated.
  flux_attn view{};
  view.cfg = *cfg;
  view.device = dev;
  if ((e = cudaDeviceGetAttribute(&view.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  view.ws = nullptr;
  view.ws_bytes = 0;
  {
    int j = 0;
    for (int a = 0; a < 3; ++a)
      for (int jj = 0; jj < ax[a] / 2; ++jj, ++j) {
        view.rope_tab.freq[j] = static_cast<float>(std::pow(static_cast<double>(cfg->rope_theta), -2.0 * jj / ax[a]));
        view.rope_tab.axis[j] = a;
      }
  }
  int n = 0;
  int rc = token_count(&view, txt_len, img_h, img_w, ref_h, ref_w, &n);
  if (rc || n == 0) return rc;
  const long long token_heads = static_cast<long long>(cfg->batch) * cfg->num_heads * n;
  if (token_heads > kNoAllocMaxTokenHeads)
    return fail(FLUX_ATTN_ERR_INVALID_ARG,
                "batch * num_heads * N = %lld exceeds the allocation-free limit of %lld (16 MiB of Q'/K' scratch)",
                token_heads, kNoAllocMaxTokenHeads);
  uint8_t* base = nullptr;
  if ((rc = noalloc_setup(dev, &base))) return rc;
  view.err = reinterpret_cast<uint32_t*>(base);
  view.qn = reinterpret_cast<__nv_bfloat16*>(base + kNoAllocWordBytes);
  view.kn = reinterpret_cast<__nv_bfloat16*>(base + kNoAllocWordBytes + token_heads * kNoAllocRowBytes);

  if ((rc = check_common(&view, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, &n)))
    return rc;
  const size_t bytes = row_bytes(&view, n);
  if ((rc = check_buffer(v, bytes, "v"))) return rc;
  if ((rc = check_buffer(out, bytes, "out"))) return rc;
  if (out == q || out == k || out == v) return fail(FLUX_ATTN_ERR_INVALID_ARG, "out aliases an input");
  if (device_error != nullptr && (rc = check_buffer(device_error, sizeof(uint32_t), "device_error"))) return rc;

  // The scratch keeps the previous call's contents: the error word must start at zero.
  e = cudaMemsetAsync(view.err, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch error word");
  rc = launch_prologue(&view, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, view.qn,
                       view.kn, n, stream);
  if (rc) return rc;
  rc = launch_attention(&view, false, view.qn, view.kn, v, nullptr, n, out, stream);
  if (rc) return rc;
  if (device_error != nullptr) {
    e = cudaMemcpyAsync(device_error, view.err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying the scratch error word");
  }
  return FLUX_ATTN_OK;
}
