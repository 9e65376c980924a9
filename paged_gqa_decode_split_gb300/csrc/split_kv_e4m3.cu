// Split-KV kernel instantiations for FP16 Q x E4M3 K/V, head dim 256.
#include "split_kv.cuh"

namespace pa {
PA_DEFINE_SPLIT_LAUNCHER(launch_split_e4m3, Fp8Fmt)
}  // namespace pa
