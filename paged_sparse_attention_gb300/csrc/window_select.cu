// Local sliding-window page selection.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.D "Page-Level Sparse
// Attention"): sparse-native models combine top-K page retrieval in their dense
// layers with local attention in their sparse layers.  The local layers need no
// scoring: the selected set is the sink pages, the `window` history pages right
// before the chunk and the chunk's own pages, the same for every KV head.  The set
// is written on the device so that it stays stream-ordered with the attention
// calls that read it (and can be captured in a CUDA graph with them).
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kWindowThreads = 128;

// block h: sel[h][0..count) = [0, sinks) U [lo, own_end), ascending
__global__ void __launch_bounds__(kWindowThreads)
    window_select_kernel(int sinks, int lo, int own_end, int32_t* __restrict__ sel,
                         int32_t* __restrict__ sel_count, int max_sel) {
  const int h = blockIdx.x;
  const int count = sinks + (own_end - lo);
  int32_t* out = sel + (size_t)h * max_sel;
  for (int i = threadIdx.x; i < count; i += kWindowThreads) out[i] = i < sinks ? i : lo + (i - sinks);
  if (threadIdx.x == 0) sel_count[h] = count;
}

}  // namespace

cudaError_t launch_window_select(const Geometry& g, int sinks, int lo, int own_end, int32_t* sel,
                                 int32_t* sel_count, int max_sel, cudaStream_t st) {
  window_select_kernel<<<g.Hkv, kWindowThreads, 0, st>>>(sinks, lo, own_end, sel, sel_count, max_sel);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
