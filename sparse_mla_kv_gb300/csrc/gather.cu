// Single-stride gather of resolved pool rows.
//
// Source: Japanese article (news.ainew.jp), section "仕組み" (How it works): whether a row sits in a
// resident page or in the hot buffer, the resolver hands back pool (HMA) row ids and the rows are
// gathered with one stride; hot pages live in the same KV tensor, so the consumer sees them as
// ordinary pages.
//
// Design: HBM-bound byte copy.  The output is a flat array of 16-byte chunks; consecutive threads
// take consecutive chunks, so every warp stores 512 contiguous bytes and reads one or two source
// rows contiguously.  blockIdx.y selects the layer; a grid-stride loop over the layer's chunks is
// unrolled so each thread keeps several 16-byte loads in flight.  Row ids are re-read per chunk
// (a broadcast within the warp, served by L1).
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

template <int CPR>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const LayerPtrs ptrs, int32_t layer_begin,
                                                                const int32_t* __restrict__ rows, int64_t n,
                                                                uint8_t* __restrict__ out, int32_t row_bytes,
                                                                int64_t num_rows, int32_t* status) {
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int lr = blockIdx.y;
  const uint8_t* __restrict__ pool = ptrs.gpu[layer_begin + lr];
  const int32_t* __restrict__ lrows = rows + (int64_t)lr * n;
  uint4* __restrict__ lout = reinterpret_cast<uint4*>(out + (int64_t)lr * n * row_bytes);
  const int64_t total = n * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += stride * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (c < total) {
        const int64_t i = c / cpr;
        const int j = (int)(c - i * cpr);
        const int row = __ldg(lrows + i);
        if (row >= 0 && row < num_rows)
          v[k] = __ldg(reinterpret_cast<const uint4*>(pool + (int64_t)row * row_bytes) + j);
        else if (row != -1)
          bad = true;
      }
    }
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      if (c < total) lout[c] = v[k];
    }
  }
  if (bad && status) *status = HS_ERR_ID_RANGE;
}

}  // namespace

cudaError_t launch_gather(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, const int32_t* rows, int64_t n,
                          uint8_t* out, int32_t row_bytes, int64_t num_rows, int32_t* status, int sms,
                          cudaStream_t s) {
  const int64_t per_layer = n * (row_bytes >> 4);
  const int64_t want = (per_layer + (int64_t)kGatherThreads * kGatherUnroll - 1) / ((int64_t)kGatherThreads * kGatherUnroll);
  // persistent-style grid: about 8 resident CTAs of 256 threads per SM, split across the layers
  int64_t cap = ((int64_t)sms * 8 + nl - 1) / nl;
  if (cap < 1) cap = 1;
  const int64_t gx = want < cap ? (want > 0 ? want : 1) : cap;
  dim3 grid((unsigned)gx, (unsigned)nl);
  if (row_bytes == 656)
    gather_kernel<41><<<grid, kGatherThreads, 0, s>>>(ptrs, layer_begin, rows, n, out, row_bytes, num_rows, status);
  else
    gather_kernel<0><<<grid, kGatherThreads, 0, s>>>(ptrs, layer_begin, rows, n, out, row_bytes, num_rows, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hs
