// Split planning, the persistent work schedule, the workspace layout and the
// E4M3 decode shared by the kernels of libpa.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

// ------------------------------------------------------------ constants --
constexpr int kTileKeys = 128;     // keys per tensor-core tile (MMA M dimension)
constexpr int kSplitTarget = 512;  // a split holds about this many keys per KV head factor before the cap
constexpr int kMaxHeadFactor = 4;  // the split floor grows with the KV head count up to this factor
constexpr int kMaxSplits = 38;     // at most this many splits per request: a quarter of the 152 SMs,
                                   // so 4, 8 or 16 long requests fill whole waves of a one-CTA-per-SM grid
constexpr int kMaxBatch = 64;
constexpr int kMaxQLen = 8;
constexpr int kMaxGroup = 8;
constexpr int kMaxRows = 64;       // G * q_len rows of one packed tile
constexpr int kPageMultiple = 16;
constexpr int kMaxCtx = 1 << 20;

// Split plan of one request of L keys over Hkv KV heads.  It depends on the
// request's length and on the packed geometry (the KV head count), never on
// the batch, so a request produces the same partials (and the merge the same
// bits) whether it runs alone or next to others.  With several KV heads a
// request already yields Hkv work items per split, so the split floor grows
// with Hkv (up to kMaxHeadFactor): fewer, longer items, less per-item cost.
// Splits are whole tiles of kTileKeys keys except the last; every split is
// non-empty.
__host__ __device__ inline void split_plan(int L, int Hkv, int& num_splits, int& chunk) {
  if (L <= 0) {
    num_splits = 0;
    chunk = 0;
    return;
  }
  const int f = Hkv < 1 ? 1 : (Hkv > kMaxHeadFactor ? kMaxHeadFactor : Hkv);
  const int target = kSplitTarget * f;
  int s0 = (L + target - 1) / target;
  s0 = s0 < 1 ? 1 : (s0 > kMaxSplits ? kMaxSplits : s0);
  int per = (L + s0 - 1) / s0;
  chunk = (per + kTileKeys - 1) / kTileKeys * kTileKeys;
  num_splits = (L + chunk - 1) / chunk;
}

// Upper bound of split_plan's count over every L <= max_ctx_len and every
// Hkv.  The count itself is not monotone in L (the split length jumps by
// whole tiles), but it never exceeds clamp(ceil(L / kSplitTarget), 1,
// kMaxSplits), which is (and which a larger head factor only lowers).
__host__ __device__ inline int max_splits_for(int max_ctx_len) {
  if (max_ctx_len <= 0) return 1;
  int s0 = (max_ctx_len + kSplitTarget - 1) / kSplitTarget;
  return s0 < 1 ? 1 : (s0 > kMaxSplits ? kMaxSplits : s0);
}

// ------------------------------------------------------------ workspace --
// [0, 4)          status word (PA_FLAG_* bits, sticky)
// [512, 768)      per-request "bad input" flags             } zero between calls:
// [768, 1024)     per-request split arrival counters        } the last CTA of a
// [1024, 1028)    next merge task (the merge phase's queue) } call resets them
// [1028, 1032)    CTAs that finished the call               } (zero at first use)
// [1280, ...)     panel_ml: float2 (m, l) [B][Hkv][S_max][R]
// [...]           panel_o : float      [B][Hkv][S_max][R][D]   (unnormalised partial O)
struct WsLayout {
  size_t ml_off, o_off, total;
};
__host__ __device__ inline WsLayout ws_layout(int B, int Hkv, int s_max, int R, int D) {
  WsLayout w;
  size_t items = (size_t)B * Hkv * (size_t)s_max * R;
  w.ml_off = 1280;
  w.o_off = (w.ml_off + items * 8 + 255) / 256 * 256;
  w.total = (w.o_off + items * (size_t)D * 4 + 255) / 256 * 256;
  return w;
}
constexpr size_t kWsBadOff = 512;      // uint32 [kMaxBatch]
constexpr size_t kWsArriveOff = 768;   // uint32 [kMaxBatch]
constexpr size_t kWsQueueOff = 1024;   // uint32
constexpr size_t kWsDoneOff = 1028;    // uint32

// ------------------------------------------------------------- schedule --
// Every CTA derives the same ordered item list from ctx_lens: requests sorted
// by split length (longest first, ties by request index), then KV head, then
// split.  CTA c executes items c, c + gridDim.x, ...  The order only balances
// work; each item's arithmetic and output slot depend on (b, g, s) alone.
struct Sched {
  int total;                 // number of items
  int order[kMaxBatch];      // request index of the o-th request in schedule order
  int first[kMaxBatch + 1];  // first item of the o-th request
  int nsplit[kMaxBatch];     // splits of request b (by request index)
  int chunk[kMaxBatch];      // split length of request b
  int len[kMaxBatch];        // validated length of request b (0 if invalid)
};

struct Item {
  int b, g, s, t0, t1, L;
};

// Called by every thread of the CTA (uses __syncthreads).  Invalid lengths
// (< 0 or > max_ctx) count as 0 and raise PA_FLAG_BAD_LENGTH once (CTA 0).
// len_t: ctx_lens[threadIdx.x] for threads below B (loaded by the caller,
// which may issue the load early), unused otherwise.
__device__ inline void sched_build(Sched& S, int len_t, int B, int Hkv, int max_ctx, uint32_t* status,
                                   uint32_t* bad) {
  int t = threadIdx.x;
  if (t < B) {
    int L = len_t;
    if (L < 0 || L > max_ctx) {
      if (blockIdx.x == 0) {
        if (status) atomicOr(status, 0x2u);
        if (bad) atomicOr(bad + t, 1u);
      }
      L = 0;
    }
    int ns, ch;
    split_plan(L, Hkv, ns, ch);
    S.len[t] = L;
    S.nsplit[t] = ns;
    S.chunk[t] = ch;
  }
  __syncthreads();
  if (t == 0) {
    for (int i = 0; i < B; ++i) S.order[i] = i;
    for (int i = 1; i < B; ++i) {  // insertion sort: chunk descending, index ascending
      int v = S.order[i], j = i - 1;
      while (j >= 0 && S.chunk[S.order[j]] < S.chunk[v]) {
        S.order[j + 1] = S.order[j];
        --j;
      }
      S.order[j + 1] = v;
    }
    int acc = 0;
    for (int o = 0; o < B; ++o) {
      S.first[o] = acc;
      acc += S.nsplit[S.order[o]] * Hkv;
    }
    S.first[B] = acc;
    S.total = acc;
  }
  __syncthreads();
}

__device__ inline Item sched_item(const Sched& S, int B, int it) {
  int o = 0;
  while (o + 1 < B && S.first[o + 1] <= it) ++o;
  int b = S.order[o];
  int local = it - S.first[o];
  int ns = S.nsplit[b];
  Item x;
  x.b = b;
  x.g = local / ns;
  x.s = local % ns;
  x.L = S.len[b];
  x.t0 = x.s * S.chunk[b];
  int e = x.t0 + S.chunk[b];
  x.t1 = e < x.L ? e : x.L;
  return x;
}

// Byte offset of key t's row (relative to the KV-head base) through the block
// table, or -1 when the page id is outside [0, num_pages).  Shared by the
// split kernels' loaders and the bookkeeping check kernel.
__device__ __forceinline__ long long kv_row_offset(const int32_t* bt_row, int t, int page_size, int num_pages,
                                                   long long page_stride, long long token_stride) {
  const int page = __ldg(bt_row + t / page_size);
  if ((unsigned)page >= (unsigned)num_pages) return -1;
  return (long long)page * page_stride + (long long)(t % page_size) * token_stride;
}

// ------------------------------------------------------------ E4M3 -> FP16 --
// Every finite E4M3 value (|x| <= 448, subnormals down to 2^-9) is exactly
// representable in FP16, so the hardware conversion is exact.  x holds four
// codes (byte 0 = lowest index); lo receives codes 0,1 and hi codes 2,3 as
// FP16x2 with the lower index in the low half.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// ------------------------------------------------------------ E5M2 -> FP16 --
// E5M2 (1 sign, 5 exponent bits with bias 15, 2 mantissa bits) has the field
// layout of the upper byte of an IEEE binary16, so code c decodes exactly to
// the FP16 bit pattern c << 8 (subnormals included).  Same packing as
// e4m3x4_to_f16x4.
__device__ __forceinline__ void e5m2x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(x, 0u, 0x1404);  // bytes: 0, code 0, 0, code 1
  hi = __byte_perm(x, 0u, 0x3424);  // bytes: 0, code 2, 0, code 3
}

}  // namespace pa
