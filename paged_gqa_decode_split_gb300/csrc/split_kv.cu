// Launch dispatch of the split-KV kernel (split_kv.cuh) by element format.
#include "split_kv.cuh"

namespace pa {

int split_smem_bytes() { return Layout<Fp8Fmt, 64>::kSmemBytes; }

cudaError_t launch_split(const SplitArgs& a, KvFormat fmt, int grid, cudaStream_t stream) {
  switch (fmt) {
    case kKvE4m3: return launch_split_e4m3(a, grid, stream);
    case kKvE5m2: return launch_split_e5m2(a, grid, stream);
    case kKvF16: return launch_split_f16(a, grid, stream);
    case kKvBf16: return launch_split_bf16_d128(a, grid, stream);
    case kKvBf16D256: return launch_split_bf16_d256(a, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
