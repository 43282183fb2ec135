// Host-only check (no kernel is launched) of the stream kernel's launch
// shape for every head count the library accepts, for each output policy:
// at least one warp and no more than the policy's maximum, shared memory
// within the kernel's limit, and no empty token part.  Built and run by
// tests/test_launch_shapes.py.
#include <cstdio>
#include "quantize_fp8.cuh"
template <class Out> int check(const char* name) {
  int bad = 0;
  for (int H = 1; H <= flux::kProMaxHeads; ++H) {
    const int W = flux::stream_warps<Out>(H);
    const size_t smem = flux::stream_smem<Out>(H);
    const int hs = Out::kParts == 1 ? H : flux::prologue_part_heads(H, Out::kParts);
    const int P = Out::kParts == 1 ? 1 : (H + hs - 1) / hs;
    const int last = H - (P - 1) * hs;
    if (W < 1 || W > Out::kWarps || smem > (size_t)flux::kProSmemBytes || smem > 227 * 1024 || last < 1 || P > Out::kParts) {
      printf("%s H=%d W=%d smem=%zu hs=%d P=%d last=%d\n", name, H, W, smem, hs, P, last);
      ++bad;
    }
  }
  printf("%s: %d bad of %d head counts; W(24)=%d smem(24)=%zu W(192)=%d smem(192)=%zu\n", name, bad, flux::kProMaxHeads,
         flux::stream_warps<Out>(24), flux::stream_smem<Out>(24), flux::stream_warps<Out>(192), flux::stream_smem<Out>(192));
  return bad;
}
int main() {
  return check<flux::Bf16Rows>("Bf16Rows") + check<flux::AmaxRows>("AmaxRows") + check<flux::E4m3Rows>("E4m3Rows");
}
