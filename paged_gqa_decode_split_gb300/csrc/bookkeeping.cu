// Bookkeeping check kernels behind pa_debug_worklist and pa_debug_gather_fp8:
// the split kernel's own device schedule and its block-table addressing,
// written out for bit-exact comparison with host restatements.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "plan.cuh"
#include "kernels.cuh"

namespace pa {

namespace {

__global__ void __launch_bounds__(64) worklist_kernel(const int32_t* ctx_lens, int B, int Hkv, int max_ctx,
                                                      int32_t* items, int32_t max_items, int32_t* count,
                                                      uint32_t* status) {
  __shared__ Sched S;
  sched_build(S, threadIdx.x < B ? ctx_lens[threadIdx.x] : 0, B, Hkv, max_ctx, status, nullptr);
  if (threadIdx.x == 0) *count = S.total;
  for (int it = threadIdx.x; it < S.total && it < max_items; it += blockDim.x) {
    const Item x = sched_item(S, B, it);
    items[4 * it + 0] = x.b;
    items[4 * it + 1] = x.g;
    items[4 * it + 2] = x.t0;
    items[4 * it + 3] = x.t1;
  }
}

__global__ void __launch_bounds__(256) gather_kernel(const uint8_t* base, long long ps, long long ts, long long hs,
                                                     const int32_t* bt, const int32_t* ctx_lens, int Hkv,
                                                     int page_size, int mpr, int num_pages, int max_ctx,
                                                     int row_bytes, uint8_t* dst) {
  const int bg = blockIdx.x;
  const int b = bg / Hkv, g = bg % Hkv;
  int L = ctx_lens[b];
  if (L < 0 || L > max_ctx) L = 0;
  const int32_t* bt_row = bt + (size_t)b * mpr;
  for (int t = blockIdx.y; t < L; t += gridDim.y) {
    const long long off = kv_row_offset(bt_row, t, page_size, num_pages, ps, ts);
    if (off < 0) continue;
    const uint8_t* src = base + (long long)g * hs + off;
    uint8_t* out = dst + ((size_t)bg * max_ctx + t) * row_bytes;
    for (int c = threadIdx.x; c < row_bytes; c += blockDim.x) out[c] = src[c];
  }
}

}  // namespace

cudaError_t launch_debug_worklist(const int32_t* ctx_lens, int B, int Hkv, int max_ctx, int32_t* items,
                                  int32_t max_items, int32_t* count, uint32_t* status, cudaStream_t stream) {
  worklist_kernel<<<1, 64, 0, stream>>>(ctx_lens, B, Hkv, max_ctx, items, max_items, count, status);
  return cudaGetLastError();
}

cudaError_t launch_debug_gather(const uint8_t* base, long long ps, long long ts, long long hs, const int32_t* bt,
                                const int32_t* ctx_lens, int B, int Hkv, int page_size, int mpr, int num_pages,
                                int max_ctx, int row_bytes, uint8_t* dst, cudaStream_t stream) {
  dim3 grid(B * Hkv, 64);
  gather_kernel<<<grid, 256, 0, stream>>>(base, ps, ts, hs, bt, ctx_lens, Hkv, page_size, mpr, num_pages, max_ctx,
                                          row_bytes, dst);
  return cudaGetLastError();
}

}  // namespace pa
