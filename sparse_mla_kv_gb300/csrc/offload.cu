// Post-forward proactive offload of completed pages, all layers in one launch, and the hot-state
// reset.
//
// Source: "vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", section "Key Architectural
// Details": proactive copying queues CPU copies of completed prefix pages while the GPU keeps
// serving them, so a GPU slot can be released under pressure without another copy; lightweight
// execution copies all sparse-MLA layers together in a single launch after the forward pass,
// ordered on the model's GPU stream.  Japanese article, section "仕組み": the GPU slot is reusable as
// soon as the copy is queued (stream order), and the CPU copy is usable once the transfer is done.
//
// Design: one launch covers every (page, layer) pair: blockIdx.y is the layer, a grid-stride loop
// walks the 16-byte chunks of all listed pages, so each warp writes 512 contiguous bytes of a host
// page (full 128-byte lines over the host link).  Loads come from HBM, stores go to the mapped
// pinned host pool.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kOffloadThreads = 256;
constexpr int kOffloadUnroll = 4;

__global__ void __launch_bounds__(kOffloadThreads) offload_kernel(const LayerPtrs ptrs, int32_t page_chunks,
                                                                  int32_t num_gpu_blocks, int32_t num_host_blocks,
                                                                  const int32_t* __restrict__ gpu_blocks,
                                                                  const int32_t* __restrict__ host_blocks, int32_t n,
                                                                  int32_t* status) {
  const int l = blockIdx.y;
  const uint4* __restrict__ src = reinterpret_cast<const uint4*>(ptrs.gpu[l]);
  uint4* __restrict__ dst = reinterpret_cast<uint4*>(ptrs.host[l]);
  const int64_t total = (int64_t)n * page_chunks;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += stride * kOffloadUnroll) {
    uint4 v[kOffloadUnroll];
    int64_t o[kOffloadUnroll];
#pragma unroll
    for (int k = 0; k < kOffloadUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      o[k] = -1;
      if (c < total) {
        const int64_t i = c / page_chunks;
        const int64_t j = c - i * page_chunks;
        const int g = __ldg(gpu_blocks + i), h = __ldg(host_blocks + i);
        if (g >= 0 && g < num_gpu_blocks && h >= 0 && h < num_host_blocks) {
          v[k] = __ldcs(src + (int64_t)g * page_chunks + j);
          o[k] = (int64_t)h * page_chunks + j;
        } else {
          bad = true;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kOffloadUnroll; ++k)
      if (o[k] >= 0) dst[o[k]] = v[k];
  }
  if (bad && status) *status = HS_ERR_TABLE_RANGE;
}

__global__ void fill_i32_kernel(int32_t* __restrict__ a, int64_t count, int32_t value) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) a[i] = value;
}

// Empties the slots of the listed requests in every group: element k of the flat range
// [groups][n][C] is slot k % C of request requests[(k / C) % n] in group k / (n * C).
__global__ void reset_requests_kernel(int32_t* __restrict__ tok, int32_t* __restrict__ stamp, int32_t groups,
                                      int32_t R, int32_t C, const int32_t* __restrict__ requests, int32_t n) {
  const int64_t total = (int64_t)groups * n * C;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += stride) {
    const int64_t s = k % C, gi = k / C;
    const int32_t r = __ldg(requests + gi % n);
    const int64_t g = gi / n;
    if (r < 0 || r >= R) continue;
    const int64_t o = (g * R + r) * C + s;
    tok[o] = -1;
    stamp[o] = -1;
  }
}

}  // namespace

cudaError_t launch_offload(const LayerPtrs& ptrs, const PoolGeom& g, const int32_t* gpu_blocks,
                           const int32_t* host_blocks, int32_t n, int32_t* status, int sms, cudaStream_t s) {
  const int32_t page_chunks = (int32_t)(((int64_t)g.page_size * g.row_bytes) >> 4);
  const int64_t per_layer = (int64_t)n * page_chunks;
  const int64_t want = (per_layer + (int64_t)kOffloadThreads * kOffloadUnroll - 1) /
                       ((int64_t)kOffloadThreads * kOffloadUnroll);
  int64_t cap = ((int64_t)sms * 8 + g.num_layers - 1) / g.num_layers;
  if (cap < 1) cap = 1;
  const int64_t gx = want < cap ? (want > 0 ? want : 1) : cap;
  dim3 grid((unsigned)gx, (unsigned)g.num_layers);
  offload_kernel<<<grid, kOffloadThreads, 0, s>>>(ptrs, page_chunks, g.num_gpu_blocks, g.num_host_blocks, gpu_blocks,
                                                  host_blocks, n, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_reset_requests(int32_t* tok, int32_t* stamp, int32_t groups, int32_t R, int32_t C,
                                  const int32_t* requests, int32_t n, int sms, cudaStream_t s) {
  const int64_t total = (int64_t)groups * n * C;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  reset_requests_kernel<<<(unsigned)blocks, 256, 0, s>>>(tok, stamp, groups, R, C, requests, n);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_fill_i32(int32_t* a, int64_t count, int32_t value, int sms, cudaStream_t s) {
  int64_t blocks = (count + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  fill_i32_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, count, value);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hs
