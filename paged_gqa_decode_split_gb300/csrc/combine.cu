// Log-sum-exp combine of the split partials, plus the bookkeeping check kernels.
//
// For one output row (request b, KV head g, packed row r = qi * G + hl) with
// splits s = 0 .. S-1 in ascending order ("perf(fa2): port decode GQA
// group-swap into d128 varlen launcher", vllm.cpp pull request #48: the
// num_splits > 1 path merges split partials with their log-sum-exp):
//   M = max_s m_s,  w_s = 2^(m_s - M),  out = scale * sum_s w_s O_s / sum_s w_s l_s
// with m in log2 units.  A row with no visible key anywhere (M = -inf), a
// request of length 0 and a request flagged by an input check all write +0.0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "plan.cuh"
#include "kernels.cuh"

namespace pa {

namespace {

static_assert(kMaxSplits <= 64, "one warp computes the split weights, two splits per lane");

template <bool BF16OUT>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  __shared__ float w_s[kMaxSplits];
  __shared__ float lsum_s;
  const int row = blockIdx.x % a.R;
  const int bg = blockIdx.x / a.R;
  const int g = bg % a.Hkv;
  const int b = bg / a.Hkv;
  const int qi = row / a.G, hl = row % a.G;
  int L = a.ctx_lens[b];
  if (L < 0 || L > a.max_ctx) L = 0;
  int ns, chunk;
  split_plan(L, ns, chunk);
  const size_t orow = (size_t)(b * a.q_len + qi) * a.Hq + g * a.G + hl;
  const size_t prow = (size_t)bg * a.s_max * a.R + row;  // panel row of split 0; split s at + s * R
  // everything above reads inputs only; the partials and the input flags come
  // from the split kernel, which may still be finishing (programmatic launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.bad != nullptr && a.bad[b] != 0u) ns = 0;
  // the partial O of every split, requested before the weights are known so
  // that the two rounds of loads overlap
  const float* o0 = a.panel_o + prow * a.D;
  const size_t sstride = (size_t)a.R * a.D;
  const int d0 = threadIdx.x;  // one thread per element d of the row (blockDim.x = D <= 256)
  float o[kMaxSplits];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) o[s] = (s < ns && d0 < a.D) ? __ldg(o0 + s * sstride + d0) : 0.f;
  // one warp, splits s and s + 32 on lane s: M = max_s m_s, w_s = 2^(m_s - M),
  // lsum = sum_s w_s l_s (a fixed reduction tree, so the bits depend on ns only)
  if (threadIdx.x < 32) {
    const int s = threadIdx.x;
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    if (s < ns) {
      const float2 ml = a.panel_ml[prow + (size_t)s * a.R];
      m0 = ml.x, l0 = ml.y;
    }
    if (s + 32 < ns) {
      const float2 ml = a.panel_ml[prow + (size_t)(s + 32) * a.R];
      m1 = ml.x, l1 = ml.y;
    }
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M);
    const float w1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - M);
    float ls = w0 * l0 + w1 * l1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (s < kMaxSplits) w_s[s] = w0;
    if (s + 32 < kMaxSplits) w_s[s + 32] = w1;
    if (s == 0) {
      lsum_s = ls;
      if (a.lse != nullptr)
        a.lse[orow] = (M == -INFINITY || !(ls > 0.f)) ? -INFINITY : (M + log2f(ls)) * 0.6931471805599453f;
    }
  }
  __syncthreads();
  const float lsum = lsum_s;
  const float scale = (a.out_scale_ptr ? __ldg(a.out_scale_ptr) : 1.0f) * a.out_scale_mul;
  if (d0 < a.D) {
    const int d = d0;
    float val = 0.f;
    if (lsum > 0.f) {
      // accumulation in ascending split order
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s) acc = (s < ns) ? fmaf(w_s[s], o[s], acc) : acc;
      val = acc / lsum * scale;
    }
    if constexpr (BF16OUT) {
      reinterpret_cast<__nv_bfloat16*>(a.out)[orow * a.D + d] = __float2bfloat16_rn(val);
    } else {
      reinterpret_cast<__half*>(a.out)[orow * a.D + d] = __float2half_rn(val);
    }
  }
}

__global__ void __launch_bounds__(64) worklist_kernel(const int32_t* ctx_lens, int B, int Hkv, int max_ctx,
                                                      int32_t* items, int32_t max_items, int32_t* count,
                                                      uint32_t* status) {
  __shared__ Sched S;
  sched_build(S, ctx_lens, B, Hkv, max_ctx, status, nullptr);
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

// Launched as a programmatic dependent of the split kernel: its blocks may
// be scheduled as the split kernel's blocks retire, and each waits
// (griddepcontrol.wait) for the split kernel's completion and memory before
// it reads a partial.
cudaError_t launch_combine(const CombineArgs& a, bool bf16_out, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hkv * a.R);
  cfg.blockDim = dim3(a.D);  // one thread per output element of the row (D <= 256)
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16_out ? cudaLaunchKernelEx(&cfg, combine_kernel<true>, a) : cudaLaunchKernelEx(&cfg, combine_kernel<false>, a);
}

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
