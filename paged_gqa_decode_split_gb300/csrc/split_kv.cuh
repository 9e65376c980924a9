#pragma once
// Split-KV paged decode / speculative-verify attention on the sm_103a tensor
// cores (tcgen05 + TMEM), for five element formats:
//   Fp8Fmt    : FP16 Q, E4M3 K/V with FP32 per-tensor scales, head_dim 256
//   E5m2Fmt   : FP16 Q, E5M2 K/V with FP32 per-tensor scales, head_dim 256
//   F16Fmt    : FP16 Q/K/V, head_dim 256
//   Bf16D256Fmt: BF16 Q/K/V, head_dim 256
//   Bf16Fmt   : BF16 Q/K/V, head_dim 128
// A staging fill is 128 keys x 256 bytes: one fill per tile for 256-byte key
// rows (8-bit D 256, 16-bit D 128), two (row bytes 0-255, then 256-511) for
// the 512-byte rows of 16-bit D 256.
//
// One work item = (request b, KV head g, split s) = keys [t0, t1) of request b.
// All G query heads x q_len verify queries of KV head g form one packed tile
// of R = G * q_len <= 64 rows, so each KV byte is fetched once per KV head
// ("perf(fa2): port decode GQA group-swap into d128 varlen launcher", vllm.cpp
// pull request #48: the query heads of one KV group share one pass over KV).
//
// The tile is computed transposed, keys on the 128-lane MMA M axis and the
// packed query rows on the N axis (N = R rounded up to 16):
//   S^T[key][row] = K'[key][:] . Q[row][:]      A = K' (TMEM), B = Q (SMEM)
//   O^T[d][row]  += V'^T[d][key] P^T[key][row]  A = V' (SMEM, MN-major), B = P (SMEM, MN-major)
// with FP32 accumulators in TMEM ("SM70 attention and quantized projection
// coverage across TP sizes", section "Scope": FP16 inputs with FP32
// accumulation for both QK and PV).  For E4M3 and E5M2, K' and V' are the
// codes decoded exactly to FP16; for BF16, K' is K and V' is V converted to FP16 so
// that P can stay FP16 in the PV product.  Each TMEM lane is one key, so the
// online softmax of a row is a reduction across lanes (warp shuffles).
//
// Warp roles (20 warps; warp w runs on sub-partition w % 4):
//   3  K loader   one thread: TMA (or the warp: TMA for pages shorter than a
//                 tile, cp.async for 8-byte aligned data) of block-table-
//                 gathered K rows, a tile at a time
//   9  V loader   the same for V
//   11 Q + QK     the packed Q tile of each item (128-byte swizzle); one
//                 thread issues the QK tcgen05.mma products
//   1  PV         one thread issues the PV tcgen05.mma products
//   4-7  K decode staging -> K' in TMEM (lane = key), the QK A operand
//   0, 8, 2, 10  V decode, key quarters 0-3: staging -> V' in a ring of
//                MN-major SMEM quarter slots
//   12-15, 16-19  softmax, two groups of four, each for half of the packed
//         rows: masking, lazy-max online softmax, P^T, row sums, O^T rescale,
//         and the item's FP32 (m, l, O) partials written to the workspace.
// Every wait is bounded (see mbar_wait); a wait that runs out aborts the CTA
// cleanly, frees TMEM and raises PA_FLAG_TIMEOUT.  A warp whose lanes all wait
// on a barrier leaves as a warp (any lane's failure ends all of them), so no
// warp-wide instruction runs with part of a warp: the decode warps finish the
// tile they are in (after an abort the data no longer matters) and vote once
// at its end, where the warp is converged; a vote at every wait costs about
// 2 % of the kernel's time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstddef>

#include "plan.cuh"
#include "ptx.cuh"
#include "kernels.cuh"

namespace pa {

namespace {

struct Fp8Fmt {
  static constexpr int D = 256;
  static constexpr int kElemBytes = 1;
  static constexpr int kFills = 1;                 // staging fills per tile
  static constexpr int kQBf16 = 0;                 // Q (and K') type of the QK product
  // the TMA loader arms a whole in-page fill before its stage is released
  // (windows always do): measured per format, faster for FP16 only
  static constexpr bool kPreArm = false;
  static __device__ __forceinline__ float score_scale(const float* k_scale) {
    // S' = q . k_code;  s * log2(e) = S' * k_scale / sqrt(256) * log2(e)
    return __ldg(k_scale) * (1.0f / 16.0f) * 1.4426950408889634f;
  }
  // 16 stored bytes (16 elements) -> 8 words of FP16x2 (K' or V' values)
  static __device__ __forceinline__ void decode16(uint4 x, uint32_t* w) {
    e4m3x4_to_f16x4(x.x, w[0], w[1]);
    e4m3x4_to_f16x4(x.y, w[2], w[3]);
    e4m3x4_to_f16x4(x.z, w[4], w[5]);
    e4m3x4_to_f16x4(x.w, w[6], w[7]);
  }
};

// E5M2 K/V: the geometry, scales and score scale of the E4M3 path; only the
// decode differs (every finite E5M2 value, |x| <= 57344, is an FP16 value)
struct E5m2Fmt : Fp8Fmt {
  static __device__ __forceinline__ void decode16(uint4 x, uint32_t* w) {
    e5m2x4_to_f16x4(x.x, w[0], w[1]);
    e5m2x4_to_f16x4(x.y, w[2], w[3]);
    e5m2x4_to_f16x4(x.z, w[4], w[5]);
    e5m2x4_to_f16x4(x.w, w[6], w[7]);
  }
};

struct Bf16Fmt {
  static constexpr int D = 128;
  static constexpr int kElemBytes = 2;
  static constexpr int kFills = 1;
  static constexpr int kQBf16 = 1;
  static constexpr bool kPreArm = false;
  static __device__ __forceinline__ float score_scale(const float*) {
    return 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
  }
  // V element pair -> FP16x2 (the PV operand type): BF16x2 word -> FP16x2
  // word (exact for |x| in [2^-14, 65504]; smaller magnitudes round to the
  // FP16 subnormal grid)
  static __device__ __forceinline__ uint32_t v2_to_h2(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// BF16 Q/K/V with head_dim 256: 512-byte key rows, two staging fills per tile
struct Bf16D256Fmt : Bf16Fmt {
  static constexpr int D = 256;
  static constexpr int kFills = 2;
  static __device__ __forceinline__ float score_scale(const float*) {
    return 1.4426950408889634f * (1.0f / 16.0f);  // log2(e) / sqrt(256)
  }
};

// FP16 Q/K/V with head_dim 256: K' and V' are the stored values
struct F16Fmt {
  static constexpr int D = 256;
  static constexpr int kElemBytes = 2;
  static constexpr int kFills = 2;
  static constexpr int kQBf16 = 0;
  static constexpr bool kPreArm = true;
  static __device__ __forceinline__ float score_scale(const float*) {
    return 1.4426950408889634f * (1.0f / 16.0f);  // log2(e) / sqrt(256)
  }
  static __device__ __forceinline__ uint32_t v2_to_h2(uint32_t w) { return w; }
};

constexpr int kChunkKeys = 32;     // one chunk = one quarter of a tile = the keys of one decode warp
constexpr int kPageSeg = 8;       // chunks whose page ids a cp.async loader lane holds in registers
constexpr int kStageBytes = kTileKeys * 256;  // one tile of 256-byte key rows (swizzled TMA and cp.async)
constexpr int kWinRowBytes = 272;             // staged window of one key (TMA windows): 8 + 256 + 8 bytes
constexpr int kStageAlloc = kTileKeys * kWinRowBytes;  // staging tile reserved for either layout
constexpr float kTau = 8.0f;       // a row's reference max moves only when a score exceeds it by 2^8
constexpr float kNoMax = -1e30f;   // reference max of a row that has seen no key (finite: 2^(s - kNoMax) never NaN)
constexpr int kThreads = 640;
constexpr int kSmemLimit = 232448; // opt-in shared memory per block on sm_103a (227 KB)
constexpr int kMaxVSlots = 8;
constexpr int kPBufs = 3;         // P^T buffers: softmax(j) writes while PV(j-1) and PV(j-2) may still read theirs
constexpr int kSoftmaxBar = 1;     // named barriers 1 and 2: the two softmax groups (0 is __syncthreads)

// TMEM column map (512 columns allocated)
constexpr uint32_t kColS = 0;     // S^T, 2 buffers of 64 columns
constexpr uint32_t kColO = 128;   // O^T, d 0..127 at +0, d 128..255 at +64; head_dim 128: two buffers
                                  // of 64 columns, item n in buffer n & 1 (its epilogue overlaps item n + 1)
constexpr uint32_t kColK = 256;   // K' operand, 2 buffers of 128 columns

struct Misc {
  uint64_t kst_full, kst_empty, vst_full, vst_empty;  // the K and V staging tiles
  uint64_t kbuf_full[2], s_full[2], vtile_full[2], p_full[kPBufs], pv_done[kPBufs];
  uint64_t q_full, q_empty, o_free[2], fin, fin_qk;
  uint32_t tmem_base;
  WaitCtl ctl;
  alignas(16) int vote[2][2][4];     // per-warp vote words of each softmax group, double-buffered
  alignas(16) float mref[kMaxRows];  // read as float4
  alignas(16) float alpha[kMaxRows];
  alignas(16) float red[4][kMaxRows];
  // merge phase: per worker (five of 128 threads) its task, the wait outcome,
  // the split weights and their weighted row sum
  int ctask[5], cok[5];
  float cw[5][kMaxSplits];
  float clsum[5];
  Sched sched;
};
static_assert(offsetof(Misc, mref) % 16 == 0, "mref is read with 16-byte loads");

// Shared memory map (offsets from a 1024-byte aligned base) for one element
// format and packed-row count NM:
//   Q    K-major Q tile, D/64 atoms of NM rows x 128 B
//   P    kPBufs P^T buffers, 128 keys x 128 B (MN-major, up to 64 rows)
//   Kst  K staging tile, 128 keys x 256 B (swizzled) or x 272 B (windows)
//   Vst  V staging tile, the same
//   V    V' ring: slots of one 32-key quarter, D/64 atoms of 32 keys x 128 B,
//        as many as fit (a quarter is released as soon as its PV MMAs finish)
template <class Fmt, int NM>
struct Layout {
  static constexpr int kQAtom = NM * 128;
  static constexpr int kQBytes = (Fmt::D / 64) * kQAtom;
  static constexpr int kVAtom = kChunkKeys * 128;
  static constexpr int kVQuarter = (Fmt::D / 64) * kVAtom;
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = kQBytes;
  static constexpr int kOffKst = kOffP + kPBufs * 16384;
  static constexpr int kOffVst = kOffKst + kStageAlloc;
  static constexpr int kOffV = kOffVst + kStageAlloc;
  static constexpr int kVFit = (kSmemLimit - kOffV - (int)sizeof(Misc) - 1024) / kVQuarter;
  static constexpr int kVSlots = kVFit < kMaxVSlots ? kVFit : kMaxVSlots;
  static constexpr int kOffMisc = kOffV + kVSlots * kVQuarter;
  static constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc) + 1024;
  static_assert(kQAtom % 1024 == 0, "Q atoms must keep the 1024-byte swizzle alignment");
  static_assert(kStageAlloc % 1024 == 0, "staging tiles must keep the 1024-byte swizzle alignment");
  static_assert(kVSlots >= 4, "the V' ring must hold a whole tile");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory map exceeds the per-block limit");
  // the merge phase stages each worker's split partials below Misc
  static_assert((kThreads / 128) * kMaxSplits * 128 * 4 <= kOffMisc, "merge staging overlaps Misc");
};

// Cross-lane reduction of n per-lane values (one per packed row) in a warp.
// Each step pairs lanes l and l^mask: while the value count is even the pair
// splits the rows and exchanges halves, otherwise it combines all of them.
// Afterwards the lane holds rows base(lane) .. base(lane)+Count-1 reduced
// over all 32 lanes.
template <int n, int mask>
struct Butterfly {
  static constexpr int Count = (n % 2 == 0) ? Butterfly<n / 2, mask / 2>::Count : Butterfly<n, mask / 2>::Count;
  static constexpr int Half = (n % 2 == 0) ? n / 2 : n;
  template <bool IsMax>
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (n % 2 == 0) {
      constexpr int h = n / 2;
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int k = 0; k < h; ++k) {
        float send = up ? v[k] : v[k + h];
        float keep = up ? v[k + h] : v[k];
        float recv = __shfl_xor_sync(0xffffffffu, send, mask);
        v[k] = IsMax ? fmaxf(keep, recv) : keep + recv;
      }
      Butterfly<h, mask / 2>::template run<IsMax>(v, lane);
    } else {
#pragma unroll
      for (int k = 0; k < n; ++k) {
        float recv = __shfl_xor_sync(0xffffffffu, v[k], mask);
        v[k] = IsMax ? fmaxf(v[k], recv) : v[k] + recv;
      }
      Butterfly<n, mask / 2>::template run<IsMax>(v, lane);
    }
  }
  // Same reduction; the first step reads src (left intact) into dst[Half].
  template <bool IsMax>
  static __device__ __forceinline__ void run_from(const float* src, float* dst, int lane) {
    if constexpr (n % 2 == 0) {
      constexpr int h = n / 2;
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int k = 0; k < h; ++k) {
        float send = up ? src[k] : src[k + h];
        float keep = up ? src[k + h] : src[k];
        float recv = __shfl_xor_sync(0xffffffffu, send, mask);
        dst[k] = IsMax ? fmaxf(keep, recv) : keep + recv;
      }
      Butterfly<h, mask / 2>::template run<IsMax>(dst, lane);
    } else {
#pragma unroll
      for (int k = 0; k < n; ++k) {
        float recv = __shfl_xor_sync(0xffffffffu, src[k], mask);
        dst[k] = IsMax ? fmaxf(src[k], recv) : src[k] + recv;
      }
      Butterfly<n, mask / 2>::template run<IsMax>(dst, lane);
    }
  }
  static __device__ __forceinline__ int base(int lane) {
    if constexpr (n % 2 == 0) {
      return ((lane & mask) ? n / 2 : 0) + Butterfly<n / 2, mask / 2>::base(lane);
    } else {
      return Butterfly<n, mask / 2>::base(lane);
    }
  }
};
template <int n>
struct Butterfly<n, 0> {
  static constexpr int Count = n;
  static constexpr int Half = n;
  template <bool IsMax>
  static __device__ __forceinline__ void run(float*, int) {}
  static __device__ __forceinline__ int base(int) { return 0; }
};

__device__ __forceinline__ uint8_t* smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ size_t panel_index(const SplitArgs& a, const Item& x) {
  return ((size_t)(x.b * a.Hkv + x.g) * a.s_max + x.s) * a.R;
}

__device__ __forceinline__ int tiles_of(const Item& x) { return (x.t1 - x.t0 + kTileKeys - 1) / kTileKeys; }

// O^T buffers: one (head_dim 256 fills the 128 columns) or two of 64 columns
// (head_dim 128), the CTA's n-th item in buffer n % kOBufs
template <class Fmt>
struct OBuf {
  static constexpr int kBufs = Fmt::D == 128 ? 2 : 1;
  static __device__ __forceinline__ uint32_t col(int n) { return kColO + 64u * (uint32_t)(n % kBufs); }
  // the epilogue of item n - kBufs released buffer n % kBufs
  static __device__ __forceinline__ uint32_t free_parity(int n) { return (uint32_t)((n / kBufs) & 1) ^ 1u; }
};

// ------------------------------------------------------------------ roles --

// Key row kk of a stage (see role_loader_tma) as 16 pieces of 16 bytes; zeros
// for keys past the split end (their stage bytes are stale or a page tail).
__device__ __forceinline__ void load_stage_row(const uint8_t* stage, int kk, bool live, uint4 (&raw)[16]) {
#pragma unroll
  for (int p = 0; p < 16; ++p)
    raw[p] = live ? *reinterpret_cast<const uint4*>(stage + (p >> 3) * 16384 + kk * 128 + (((p & 7) ^ (kk & 7)) << 4))
                  : make_uint4(0u, 0u, 0u, 0u);
}

// The same from a window-layout stage (kKvLoadWindow): key kk's window at
// kk*272 holds its 256 row bytes at window bytes 8..263, so 16-byte piece p
// is the upper half of window granule p and the lower half of granule p + 1.
// Eight consecutive keys read granule g at (17kk + g) mod 8 of the 16-byte
// bank groups: all different, so no bank conflicts.
__device__ __forceinline__ void load_window_row(const uint8_t* stage, int kk, bool live, uint4 (&raw)[16]) {
  const uint8_t* row = stage + kk * kWinRowBytes;
  uint4 lo = live ? *reinterpret_cast<const uint4*>(row) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const uint4 hi = live ? *reinterpret_cast<const uint4*>(row + 16 * (p + 1)) : make_uint4(0u, 0u, 0u, 0u);
    raw[p] = make_uint4(lo.z, lo.w, hi.x, hi.y);
    lo = hi;
  }
}

template <bool Win>
__device__ __forceinline__ void load_row(const uint8_t* stage, int kk, bool live, uint4 (&raw)[16]) {
  if constexpr (Win) {
    load_window_row(stage, kk, live, raw);
  } else {
    load_stage_row(stage, kk, live, raw);
  }
}

// K and V loaders: one tile (128 keys) at a time into the tensor's staging
// tile.  Layout: two halves of the 256-byte key rows, half h at h*16384, key
// kk's 128 bytes at kk*128 with its 16-byte piece p at ((p ^ (kk & 7)) * 16)
// (the TMA 128-byte swizzle), so the decode warps read eight consecutive keys
// without bank conflicts.  The tile is refilled once all four decode warps
// have copied their rows out.  Keys past the split end may hold anything; the
// decode warps zero them.

// Block-table entry, loaded where it stands in the program (not sunk to its
// first use), so that the loader can fetch page ids ahead of need.
__device__ __forceinline__ int ld_page_id(const int32_t* p) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// TMA mode (16-byte aligned bases and strides): one thread.  A tile inside
// one page is one copy: a box of the 5-D byte view (row byte 0..127, KV head,
// slot, 128-byte part of the row, page) that writes both halves.  Otherwise
// the tile's keys are cut at page boundaries; each piece (a multiple of 16
// slots inside one page) is covered by boxes of 128, 64, 32 and 16 slots of
// the 4-D byte view (row byte, KV head, slot, page), two boxes (row bytes
// 0-127 and 128-255) per piece of slots.  Window mode (Win, bases 8 bytes
// past a 16-byte boundary): one box of 272-byte windows per piece of slots
// (a whole in-page tile is one box of 128 slots), each key's window at
// kk*272 of the stage.  Completion is
// counted in bytes on the tile's full barrier; the thread arrives with the
// byte total after issuing the copies.  Page ids are kept for the current
// page index and the three after it, each loaded several pages ahead.  The
// thread issues few instructions per tile: the shared per-SM instruction
// queues are busy with the decode warps' traffic.  With two fills per tile
// (512-byte rows) the pieces are walked twice, fill h copying row bytes
// 256h .. 256h+255.
template <class Fmt, bool Win>
__device__ __forceinline__ void role_loader_tma(const SplitArgs& a, Misc& M, bool is_v, uint8_t* stage) {
  const CUtensorMap* maps = is_v ? a.v_maps : a.k_maps;  // boxes of 128, 64, 32, 16 slots
  const CUtensorMap* tile_map = is_v ? &a.v_map_tile : &a.k_map_tile;  // 128 slots x both parts
  uint64_t* full = is_v ? &M.vst_full : &M.kst_full;
  uint64_t* empty = is_v ? &M.vst_empty : &M.kst_empty;
  WaitCtl* abort = &M.ctl;
  const int ps = a.page_size;
  const uint32_t dst_base = smem_u32(stage);
  // K and V are read once per call: evict them from L2 first, so that the
  // split partials the merge phase reads at the end of the grid stay resident
  const uint64_t once = l2_policy_evict_first();
  uint32_t f = 0;  // fills issued
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int32_t* bt = a.block_table + (size_t)x.b * a.mpr;
    const int nt = tiles_of(x);
    const int q_last = (x.t1 - 1) / ps;  // last page index the item reads
    int q_cur = x.t0 / ps;
    int pq[4];                           // page ids of page indices q_cur .. q_cur+3 (-1 past q_last)
#pragma unroll
    for (int k = 0; k < 4; ++k) pq[k] = q_cur + k <= q_last ? ld_page_id(bt + q_cur + k) : -1;
    for (int jl = 0; jl < nt; ++jl) {
      const int kb = x.t0 + jl * kTileKeys;
      const int rows = (min(kb + kTileKeys, x.t1) - kb + 15) & ~15;  // whole 16-key blocks holding split keys
      const int q_tile = q_cur;
      const int pq_tile[4] = {pq[0], pq[1], pq[2], pq[3]};
#pragma unroll
      for (int h = 0; h < Fmt::kFills; ++h, ++f) {
        if (h > 0) {  // walk the tile's pages again for the next 256 row bytes
          q_cur = q_tile;
#pragma unroll
          for (int k = 0; k < 4; ++k) pq[k] = pq_tile[k];
        }
        // Windows and FP16 tiles: the fill's first piece is located before the
        // stage is free.  A whole tile inside one page is one box, and its byte
        // count is armed on the full barrier as soon as the previous fill has
        // landed (the phase then waits for the bytes alone), so that once the
        // decode warps release the stage only the copy itself is left to issue.
        // The other 16-byte aligned formats measured slower with this order and
        // take the general path below.
        constexpr bool kPreArm = Win || Fmt::kPreArm;
        bool whole = false;
        int slot0 = 0, pg0 = -1;
        if constexpr (kPreArm) {
          const int q0 = kb / ps;
          slot0 = kb - q0 * ps;
          for (int adv = 0; adv < kTileKeys / 16 && q_cur < q0; ++adv) {
            pq[0] = pq[1], pq[1] = pq[2], pq[2] = pq[3];
            ++q_cur;
            pq[3] = q_cur + 3 <= q_last ? ld_page_id(bt + q_cur + 3) : -1;
          }
          pg0 = pq[0];
          whole = rows == kTileKeys && slot0 + kTileKeys <= ps && (unsigned)pg0 < (unsigned)a.num_pages;
          if (whole) {
            if (f > 0 && !mbar_wait(full, (f - 1) & 1, abort)) {
              mbar_drain(full, (f - 1) & 1, abort);
              return;
            }
            mbar_arrive_expect_tx(full, Win ? kTileKeys * kWinRowBytes : kTileKeys * 256);
          }
        }
        if (!mbar_wait(empty, (f & 1) ^ 1, abort)) {
          // fill f - 1 may still be landing: let it finish before the CTA exits
          if (f > 0) mbar_drain(full, (f - 1) & 1, abort);
          return;
        }
        if (whole) {
          if constexpr (Win) {
            // window element 128h is the byte 8 before row byte 256h
            tma_load_4d_hint(dst_base, maps, 128 * h, x.g, slot0, pg0, full, once);
          } else {
            tma_load_5d_hint(dst_base, tile_map, 0, x.g, slot0, 2 * h, pg0, full, once);
          }
          continue;
        }
        uint32_t bytes = 0;
        bool bad = false;
        for (int r = 0; r < rows;) {
          const int t = kb + r;
          const int q = t / ps;
          const int slot = t - q * ps;
          const int len = min(rows - r, ps - slot);  // a multiple of 16
          for (int adv = 0; adv < kTileKeys / 16 && q_cur < q; ++adv) {
            pq[0] = pq[1], pq[1] = pq[2], pq[2] = pq[3];
            ++q_cur;
            pq[3] = q_cur + 3 <= q_last ? ld_page_id(bt + q_cur + 3) : -1;
          }
          const int pg = pq[0];
          if constexpr (Win) {
            if ((unsigned)pg < (unsigned)a.num_pages) {
              // window element 128h is the byte 8 before row byte 256h
              int rr = r, sl = slot, left = len;
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int box = kTileKeys >> m;  // 128, 64, 32, 16 slots
                while (left >= box) {
                  tma_load_4d_hint(dst_base + rr * kWinRowBytes, maps + m, 128 * h, x.g, sl, pg, full, once);
                  bytes += box * kWinRowBytes;
                  rr += box, sl += box, left -= box;
                }
              }
            } else {
              bad = true;
            }
          } else if ((unsigned)pg < (unsigned)a.num_pages && len == kTileKeys) {
            // the whole tile inside one page: one box writes both parts
            tma_load_5d_hint(dst_base, tile_map, 0, x.g, slot, 2 * h, pg, full, once);
            bytes += kTileKeys * 256;
          } else if ((unsigned)pg < (unsigned)a.num_pages) {
            int rr = r, sl = slot, left = len;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int box = kTileKeys >> m;  // 128, 64, 32, 16 slots
              while (left >= box) {
                tma_load_4d_hint(dst_base + rr * 128, maps + m, 256 * h, x.g, sl, pg, full, once);
                tma_load_4d_hint(dst_base + 16384 + rr * 128, maps + m, 256 * h + 128, x.g, sl, pg, full, once);
                bytes += box * 256;
                rr += box, sl += box, left -= box;
              }
            }
          } else {
            bad = true;
          }
          r += len;
        }
        if (bad) {
          atomicOr(a.status, 0x1u);
          atomicOr(a.bad + x.b, 1u);
        }
        mbar_arrive_expect_tx(full, bytes);
      }
    }
  }
}

// TMA mode for pages shorter than a tile (page_size < 128, so a tile spans
// several pages): the whole loader warp.  Lane l < 8 owns the tile's 16-key
// block l, which never straddles a page (page sizes are multiples of 16), and
// issues its two 16-slot boxes (row bytes 0-127 and 128-255 of the fill), so
// the eight pieces of a tile are issued by one warp instruction instead of
// one after another by a single thread.  Each lane loads its block's page id
// a tile ahead.  Lane 0 waits for the staging tile and arrives with the byte
// total once the warp has issued.
template <class Fmt>
__device__ __forceinline__ void role_loader_tma_blocks(const SplitArgs& a, Misc& M, bool is_v, uint8_t* stage,
                                                       int lane) {
  constexpr int kBlocks = kTileKeys / 16;
  const CUtensorMap* map16 = (is_v ? a.v_maps : a.k_maps) + 3;  // boxes of 16 slots
  uint64_t* full = is_v ? &M.vst_full : &M.kst_full;
  uint64_t* empty = is_v ? &M.vst_empty : &M.kst_empty;
  WaitCtl* abort = &M.ctl;
  const int ps = a.page_size;
  const uint32_t dst = smem_u32(stage) + 16 * lane * 128;
  const uint64_t once = l2_policy_evict_first();  // K and V are read once per call
  uint32_t f = 0;  // fills issued
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int32_t* bt = a.block_table + (size_t)x.b * a.mpr;
    const int nt = tiles_of(x);
    // first key of this lane's block of tile jl, and whether it holds split keys
    auto block_key = [&](int jl) { return x.t0 + jl * kTileKeys + 16 * lane; };
    auto block_live = [&](int jl) { return lane < kBlocks && jl < nt && block_key(jl) < x.t1; };
    int pg_next = block_live(0) ? ld_page_id(bt + block_key(0) / ps) : -1;
    for (int jl = 0; jl < nt; ++jl) {
      const int pg = pg_next;
      pg_next = block_live(jl + 1) ? ld_page_id(bt + block_key(jl + 1) / ps) : -1;
      const bool live = block_live(jl);
      const bool ok = live && (unsigned)pg < (unsigned)a.num_pages;
      if (live && !ok) {
        atomicOr(a.status, 0x1u);
        atomicOr(a.bad + x.b, 1u);
      }
      const int slot = block_key(jl) % ps;
      const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, ok)) * 16u * 256u;
#pragma unroll
      for (int h = 0; h < Fmt::kFills; ++h, ++f) {
        int go = 1;
        if (lane == 0) {
          go = mbar_wait(empty, (f & 1) ^ 1, abort) ? 1 : 0;
          // fill f - 1 may still be landing: let it finish before the CTA exits
          if (!go && f > 0) mbar_drain(full, (f - 1) & 1, abort);
        }
        if (__shfl_sync(0xffffffffu, go, 0) == 0) return;
        if (ok) {
          tma_load_4d_hint(dst, map16, 256 * h, x.g, slot, pg, full, once);
          tma_load_4d_hint(dst + 16384, map16, 256 * h + 128, x.g, slot, pg, full, once);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(full, bytes);
      }
    }
  }
}

// cp.async mode (8-byte aligned data): every lane copies 8-byte pieces of
// the tile's rows into the same layout, zero-filling rows past the split end,
// 32 keys at a time.  Lane l holds the page ids of key t0 + 32*cj + l for
// eight 32-key chunks at a time: `cur` serves chunks cs..cs+7 while `nxt` is
// being loaded for cs+8..cs+15.
template <class Fmt>
__device__ __forceinline__ void role_loader_cp(const SplitArgs& a, Misc& M, bool is_v, int lane, uint8_t* stage) {
  const uint8_t* base = is_v ? a.v : a.k;
  const long long pstr = is_v ? a.v_ps : a.k_ps;
  const long long tstr = is_v ? a.v_ts : a.k_ts;
  const long long hstr = is_v ? a.v_hs : a.k_hs;
  uint64_t* full = is_v ? &M.vst_full : &M.kst_full;
  uint64_t* empty = is_v ? &M.vst_empty : &M.kst_empty;
  WaitCtl* abort = &M.ctl;
  const uint32_t dst_base = smem_u32(stage);
  uint32_t f = 0;  // fills issued
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int32_t* bt = a.block_table + (size_t)x.b * a.mpr;
    const uint8_t* hbase = base + (long long)x.g * hstr;
    const int nchunks = tiles_of(x) * (kTileKeys / kChunkKeys);
    auto load_segment = [&](int (&pg)[kPageSeg], int cs) {
#pragma unroll
      for (int s = 0; s < kPageSeg; ++s) {
        const int cj = cs + s;
        const int t = x.t0 + cj * kChunkKeys + lane;
        pg[s] = (cj < nchunks && t < x.t1) ? ld_page_id(bt + t / a.page_size) : -1;
      }
    };
    int cur[kPageSeg], nxt[kPageSeg];
    load_segment(cur, 0);
    load_segment(nxt, kPageSeg);
    for (int cs = 0; cs < nchunks; cs += kPageSeg) {
      // the segment's tiles (four chunks each); per tile one fill of each 256
      // row bytes
#pragma unroll
      for (int tq = 0; tq < kPageSeg / 4; ++tq) {
        if (cs + 4 * tq >= nchunks) break;
#pragma unroll
        for (int h = 0; h < Fmt::kFills; ++h, ++f) {
          if (!mbar_wait(empty, (f & 1) ^ 1, abort)) goto done;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // quarter of the tile
            const int s = 4 * tq + q4;
            const int page_cur = cur[s];
            const int kb = x.t0 + (cs + s) * kChunkKeys;
            const int t = kb + lane;
            long long rowoff = -1;
            if (t < x.t1) {
              if ((unsigned)page_cur < (unsigned)a.num_pages) {
                rowoff = (long long)page_cur * pstr + (long long)(t % a.page_size) * tstr + 256 * h;
              } else if (h == 0) {
                atomicOr(a.status, 0x1u);
                atomicOr(a.bad + x.b, 1u);
              }
            }
#pragma unroll 4
            for (int kq = 0; kq < kChunkKeys; ++kq) {
              const long long ro = __shfl_sync(0xffffffffu, rowoff, kq);
              const int kk = 32 * q4 + kq;  // key of the tile
              const int piece = lane >> 1;  // 16-byte piece 0..15 of the fill's 256 row bytes
              const uint8_t* src = ro >= 0 ? hbase + ro + lane * 8 : base;
              const uint32_t dst =
                  dst_base + (piece >> 3) * 16384 + kk * 128 + (((piece & 7) ^ (kk & 7)) << 4) + (lane & 1) * 8;
              cp_async_8(dst, src, ro >= 0 ? 8u : 0u);
            }
          }
          cp_async_arrive(full);
        }
      }
#pragma unroll
      for (int s = 0; s < kPageSeg; ++s) cur[s] = nxt[s];
      load_segment(nxt, cs + 2 * kPageSeg);
    }
  }
done:
  cp_async_wait_all();
}

// Q tile and QK issuer (one warp): per item the warp loads the packed Q tile
// (row r = qi * G + hl holds query head g*G + hl of verify query qi; K-major,
// element (r, d) at (d/64)*(NM*128) + r*128 + ((((d%64)/8) ^ (r%8)) * 16) +
// (d%8)*2) once every QK of the previous item completed (q_empty): one TMA box
// per 64-column atom (the 128-byte swizzle of the copy is this layout) when
// K and V are loaded by TMA as well, else 16-byte copies by every lane; lane 0 then
// issues QK(j) for the item's tiles (S^T[128 keys x N] = K' Q^T, 16 steps of
// K = 16, FP32 in TMEM), each once K'(j) is written and S[j&1] is free (the
// softmax signalled P^T(j-2) after its last read of it), and commits to
// s_full (which also frees K'[j&1]); an item's last QK also to q_empty.  The
// PV products come from another thread (role_pv), so that neither stream of
// tensor-core work waits behind the other's dependencies.
template <class Fmt, int NM>
__device__ __forceinline__ void role_q_qk(const SplitArgs& a, Misc& M, int lane, uint8_t* qbuf, uint32_t tb) {
  using L = Layout<Fmt, NM>;
  constexpr int kPieces = Fmt::D / 8;
  constexpr uint32_t id_qk = idesc_f16(128, NM, Fmt::kQBf16, 0, 0);
  constexpr int kKSteps = Fmt::D / 16;
  WaitCtl* abort = &M.ctl;
  const uint16_t* q = reinterpret_cast<const uint16_t*>(a.q);
  const uint64_t q_desc = sdesc_sw128(smem_u32(qbuf), 16, 1024);
  uint32_t j = 0;
  bool ok = true;
  for (int it = blockIdx.x, n = 0; ok && it < M.sched.total; it += gridDim.x, ++n) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    if (!__all_sync(0xffffffffu, mbar_wait(&M.q_empty, (n & 1) ^ 1, abort))) break;
    if (a.q_tma) {
      // one box per 64-column atom: rows (qi, hl) land at r = qi * G + hl
      if (lane == 0 && !a.withhold_q) {  // withheld only by the timeout test hook
#pragma unroll
        for (int c = 0; c < Fmt::D / 64; ++c)
          tma_load_4d(smem_u32(qbuf + c * L::kQAtom), &a.q_map, 64 * c, x.g * a.G, 0, x.b, &M.q_full);
        mbar_arrive_expect_tx(&M.q_full, (uint32_t)((Fmt::D / 64) * a.R * 128));
      }
    } else {
      for (int u = lane; u < a.R * kPieces; u += 32) {
        const int r = u / kPieces, c = u % kPieces;
        const int qi = r / a.G, hl = r % a.G;
        const uint16_t* src = q + ((size_t)(x.b * a.q_len + qi) * a.Hq + x.g * a.G + hl) * Fmt::D + c * 8;
        const uint32_t dst = smem_u32(qbuf + (c >> 3) * (NM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
        cp_async_16(dst, src, 16u);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && !a.withhold_q) mbar_arrive(&M.q_full);
    }
    // the next item's Q rows into L2, so that its Q tile is not a round trip
    // to HBM at the item boundary (each row is D * 2 bytes of one query head)
    if (it + (int)gridDim.x < M.sched.total) {
      const Item y = sched_item(M.sched, a.B, it + gridDim.x);
      for (int u = lane; u < a.R * (Fmt::D * 2 / 128); u += 32) {
        const int r = u / (Fmt::D * 2 / 128), l = u % (Fmt::D * 2 / 128);
        const int qi = r / a.G, hl = r % a.G;
        prefetch_l2(q + ((size_t)(y.b * a.q_len + qi) * a.Hq + y.g * a.G + hl) * Fmt::D + l * 64);
      }
    }
    if (lane == 0) {
      ok = mbar_wait(&M.q_full, n & 1, abort);
      // an abort while this item's Q boxes are in flight: let them land
      if (!ok && a.q_tma && !a.withhold_q) mbar_drain(&M.q_full, n & 1, abort);
      for (int jl = 0; ok && jl < nt; ++jl, ++j) {
        if (j >= 2) ok = mbar_wait(&M.p_full[(j - 2) % kPBufs], ((j - 2) / kPBufs) & 1, abort);
        ok = ok && mbar_wait(&M.kbuf_full[j & 1], (j >> 1) & 1, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = tb + kColS + (j & 1) * 64, k_col = tb + kColK + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk)
          mma_ts(s_col, k_col + kk * 8, sdesc_add(q_desc, (kk >> 2) * L::kQAtom + (kk & 3) * 32), id_qk,
                 kk > 0 ? 1u : 0u);
        mma_commit(&M.s_full[j & 1]);
        if (jl == nt - 1) mma_commit(&M.q_empty);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  cp_async_wait_all();
}

// K decode: warp quarter i owns TMEM lanes 32i..32i+31 = keys 32i.. of each
// tile; lane = key, column c holds elements d = 2c, 2c+1.  With two staging
// fills per tile, fill h supplies columns 64h .. 64h+63.
template <class Fmt, bool Win>
__device__ __forceinline__ void role_kdecode(const SplitArgs& a, Misc& M, int i, int lane, uint32_t tb,
                                             const uint8_t* stage) {
  WaitCtl* abort = &M.ctl;
  uint32_t j = 0, f = 0;  // tiles, staging fills
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    for (int jl = 0; jl < nt; ++jl, ++j) {
      bool ok = true;  // every wait of this tile succeeded (the warp decides at the tile's end)
#pragma unroll
      for (int h = 0; h < Fmt::kFills; ++h, ++f) {
        ok = mbar_wait(&M.kst_full, f & 1, abort) && ok;
        // take this key's 256 staged row bytes into registers and hand the
        // stage back at once, so the loader's refill does not wait for the
        // tensor core
        uint4 raw[16];
        load_row<Win>(stage, 32 * i + lane, x.t0 + jl * kTileKeys + 32 * i + lane < x.t1, raw);
        // the row reads (generic proxy) are ordered before the next fill,
        // which the TMA writes through the async proxy once the stage is free
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.kst_empty);
        // K'[j&1] is free once QK(j-2) is done (its completion is s_full's phase)
        if (h == 0 && j >= 2) ok = mbar_wait(&M.s_full[j & 1], ((j >> 1) & 1) ^ 1, abort) && ok;
        const uint32_t taddr = tb + ((uint32_t)(32 * i) << 16) + kColK + (j & 1) * 128 + h * 64;
        if constexpr (Fmt::kElemBytes == 1) {
#pragma unroll
          for (int c2 = 0; c2 < 8; ++c2) {
            uint32_t r[16];
            Fmt::decode16(raw[2 * c2], r);
            Fmt::decode16(raw[2 * c2 + 1], r + 8);
            PA_TMEM_ST_X16(taddr + c2 * 16, r);
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t r[16];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint4 w = raw[4 * c4 + e];
              r[4 * e + 0] = w.x, r[4 * e + 1] = w.y, r[4 * e + 2] = w.z, r[4 * e + 3] = w.w;
            }
            PA_TMEM_ST_X16(taddr + c4 * 16, r);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.kbuf_full[j & 1]);
      if (__any_sync(0xffffffffu, !ok)) return;
    }
  }
}

// V decode: warp quarter i converts keys 32i.. of each tile, i.e. quarter
// c = 4j + i of the CTA's key sequence, into slot c % kVSlots of the V' ring.
// MN-major V' operand: element (key kq of the quarter, d) at (d/64)*4096 +
// kq*128 + ((((d%64)/8) ^ (kq%8)) * 16) + (d%8)*2.  A slot is rewritten once
// the PV of the tile that read its previous quarter has completed; the four
// warps signal the tile's quarters on one barrier.
template <class Fmt, int NM, bool Win>
__device__ __forceinline__ void role_vdecode(const SplitArgs& a, Misc& M, int i, int lane, const uint8_t* stage,
                                             uint8_t* vring) {
  using L = Layout<Fmt, NM>;
  WaitCtl* abort = &M.ctl;
  uint32_t j = 0, f = 0;  // tiles, staging fills
  const int key = 32 * i + lane;
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    for (int jl = 0; jl < nt; ++jl, ++j) {
      const uint32_t c = 4 * j + i;
      const int slot = (int)(c % L::kVSlots);
      bool ok = true;  // every wait of this tile succeeded (the warp decides at the tile's end)
#pragma unroll
      for (int h = 0; h < Fmt::kFills; ++h, ++f) {
        ok = mbar_wait(&M.vst_full, f & 1, abort) && ok;
        // row into registers, stage back to the loader, then wait for the slot
        uint4 raw[16];
        load_row<Win>(stage, key, x.t0 + jl * kTileKeys + key < x.t1, raw);
        fence_proxy_async_smem();  // the row reads before the next fill's TMA writes
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.vst_empty);
        if (h == 0 && c >= (uint32_t)L::kVSlots) {
          // the slot's previous quarter belongs to tile t; PV(t) done frees it
          const uint32_t t = (c - L::kVSlots) / 4;
          ok = mbar_wait(&M.pv_done[t % kPBufs], (t / kPBufs) & 1, abort) && ok;
        }
        uint8_t* dst0 = vring + slot * L::kVQuarter + lane * 128;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint4 x4 = raw[ch];
          if constexpr (Fmt::kElemBytes == 1) {
            // piece ch = d 16ch .. 16ch+15 -> two 8-element FP16 pieces
            uint32_t w[8];
            Fmt::decode16(x4, w);
            const int at = ch >> 2, u = ch & 3;
            uint8_t* dst = dst0 + at * L::kVAtom;
            *reinterpret_cast<uint4*>(dst + (((2 * u) ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + (((2 * u + 1) ^ (lane & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            // piece ch of fill h = d 128h + 8ch .. 128h + 8ch + 7
            const uint4 w = make_uint4(Fmt::v2_to_h2(x4.x), Fmt::v2_to_h2(x4.y), Fmt::v2_to_h2(x4.z),
                                       Fmt::v2_to_h2(x4.w));
            const int at = 2 * h + (ch >> 3), u = ch & 7;
            *reinterpret_cast<uint4*>(dst0 + at * L::kVAtom + ((u ^ (lane & 7)) << 4)) = w;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.vtile_full[j & 1]);
      if (__any_sync(0xffffffffu, !ok)) return;
    }
  }
}

// PV issuer (one thread): for every tile j, once the softmax has written
// P^T(j) and the V decode warps V'(j) (on an item's first tile also once the
// epilogue released O): O^T[d x N] += V'^T P^T over the tile's four V' slots
// (2 halves of M 128 x 8 steps of K = 16), committed to pv_done (which also
// frees P^T(j) and the V' slots of tile j).  Operand descriptors are built
// once and advanced by compile-time offsets.
template <class Fmt, int NM>
__device__ __forceinline__ void role_pv(const SplitArgs& a, Misc& M, uint32_t tb, uint32_t pbase, uint32_t vbase) {
  using L = Layout<Fmt, NM>;
  constexpr uint32_t id_pv = idesc_f16(128, NM, 0, 1, 1);
  constexpr int kHalves = Fmt::D / 128;
  WaitCtl* abort = &M.ctl;
  const uint64_t v_desc = sdesc_sw128(vbase, L::kVAtom, 1024);
  const uint64_t p_desc = sdesc_sw128(pbase, 16384, 1024);
  uint32_t pj = 0;
  int slot0 = 0;
  for (int n = 0, it = blockIdx.x; it < M.sched.total; ++n, it += gridDim.x) {
    const int nt = tiles_of(sched_item(M.sched, a.B, it));
    for (int jl = 0; jl < nt; ++jl, ++pj) {
      const uint32_t pb = pj % kPBufs, pu = pj / kPBufs;
      if (!mbar_wait(&M.p_full[pb], pu & 1, abort)) return;
      if (jl == 0 && !mbar_wait(&M.o_free[n % OBuf<Fmt>::kBufs], OBuf<Fmt>::free_parity(n), abort)) return;
      if (!mbar_wait(&M.vtile_full[pj & 1], (pj >> 1) & 1, abort)) return;
      tc_fence_after();
      const uint64_t pd = sdesc_add(p_desc, pb * 16384);
      const uint32_t first = jl == 0 ? 0u : 1u;
      int slot = slot0;
#pragma unroll
      for (int pq = 0; pq < 4; ++pq) {
        const uint64_t vd = sdesc_add(v_desc, slot * L::kVQuarter);
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_ss(tb + OBuf<Fmt>::col(n) + 64 * h, sdesc_add(vd, 2 * h * L::kVAtom + kk * 2048),
                   sdesc_add(pd, (2 * pq + kk) * 2048), id_pv, (pq == 0 && kk == 0) ? first : 1u);
        }
        slot = slot + 1 == L::kVSlots ? 0 : slot + 1;
      }
      slot0 = slot;
      mma_commit(&M.pv_done[pb]);
    }
  }
}

// Softmax warps: two groups of four; group grp owns packed rows
// [grp*RG, (grp+1)*RG) with RG = NM/2, and warp quarter i of a group reads
// TMEM lanes 32i.. (keys of S^T, then d of O^T) of the group's columns.  The
// groups never synchronise with each other: every row's running state lives
// in one group.
//
// Scores stay in S units (the raw QK^T accumulator); c = log2(e) * scale turns
// them into the log2 domain inside one FFMA.  Per row r the group keeps a
// reference max m_r (log2 units; kNoMax before any visible key).  One pass per
// tile over the group's rows: x = S*c - m_r; a vote of the group's four warps
// (a named barrier) checks x <= tau for every visible score, and then P = 2^x
// is written as FP16 (at most 2^tau) with no cross-lane reduction.  A tile
// whose vote fails takes the row maxima of the tile, moves the references,
// rescales the row sums and the O^T columns of those rows, and recomputes x.
// Each thread keeps the running row sums of its own key slot for the group's
// rows, reduced once per item.  Every wait is bounded; a wait that runs out
// is reported through the next vote, so the group's warps always leave
// together and never strand one another at a barrier.
template <class Fmt, int NM>
__device__ __forceinline__ void role_softmax(const SplitArgs& a, Misc& M, int grp, int i, int lane, uint32_t tb,
                                             uint8_t* pbuf) {
  constexpr int RG = NM / 2;  // rows of the group, a multiple of 8
  using BF = Butterfly<RG, 16>;
  constexpr int CNT = BF::Count;
  constexpr int kHalves = Fmt::D / 128;
  WaitCtl* abort = &M.ctl;
  const int gt = 32 * i + lane;  // thread index inside the group = key of the tile
  const int row0 = grp * RG;
  const int bar_id = kSoftmaxBar + grp;
  const float c_log2 = Fmt::score_scale(a.k_scale);
  const uint32_t lane_base = tb + ((uint32_t)(32 * i) << 16);
  // the split partials are read back by the merge phase at the end of this
  // grid: keep their L2 lines
  const uint64_t keep = l2_policy_evict_last();
  const int rbase = BF::base(lane);  // rows row0+rbase .. +CNT-1 of every butterfly result
  uint32_t j = 0, nvote = 0;
  bool bad = false;
  // returns bit 0: some warp saw an exceeding score, bit 1: some wait ran out
  auto vote = [&](bool ex) -> int {
    const int f = (__any_sync(0xffffffffu, ex) ? 1 : 0) | (__any_sync(0xffffffffu, bad) ? 2 : 0);
    int* slot = M.vote[grp][nvote & 1];
    ++nvote;
    if (lane == 0) slot[i] = f;
    named_bar_sync(bar_id, 128);
    const int4 w = *reinterpret_cast<const int4*>(slot);
    return w.x | w.y | w.z | w.w;
  };
  // RG consecutive TMEM columns of this thread's lane
  auto tmem_load_rows = [&](uint32_t addr, uint32_t (&r)[RG]) {
#pragma unroll
    for (int c = 0; c < RG / 8; ++c) PA_TMEM_LD_X8(addr + 8 * c, r + 8 * c);
    tmem_wait_ld();
    reg_fence(r);
  };
  for (int it = blockIdx.x, n = 0; it < M.sched.total; it += gridDim.x, ++n) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    const uint32_t ocol = OBuf<Fmt>::col(n);  // this item's O^T columns
    const int lim = x.L - a.q_len;  // packed row r sees key t iff t <= lim + r / G
    float lsum[RG];                 // running row sums of this thread's key slot
#pragma unroll
    for (int r = 0; r < RG; ++r) lsum[r] = 0.f;
    for (int jl = 0; jl < nt; ++jl, ++j) {
      bad |= !mbar_wait(&M.s_full[j & 1], (j >> 1) & 1, abort);
      // P^T buffer j % kPBufs is free once PV(j - kPBufs) is done
      const uint32_t pb = j % kPBufs;
      if (j >= kPBufs) bad |= !mbar_wait(&M.pv_done[pb], ((j / kPBufs) - 1) & 1, abort);
      tc_fence_after();
      const uint32_t s_addr = lane_base + kColS + (j & 1) * 64 + row0;
      const int tile0 = x.t0 + jl * kTileKeys;
      const int key = tile0 + gt;
      const int vis_end = min(x.t1, lim + 1);  // keys below this are visible to every row
      const bool masked_tile = tile0 + kTileKeys > vis_end || NM > a.R;
      uint8_t* prow = pbuf + pb * 16384 + gt * 128;
      // the group's scores of this key, masked to -inf where invisible
      auto load_scores = [&](float (&v)[RG]) {
        uint32_t r[RG];
        tmem_load_rows(s_addr, r);
#pragma unroll
        for (int k = 0; k < RG; ++k) v[k] = __uint_as_float(r[k]);
        if (masked_tile) {
#pragma unroll
          for (int k = 0; k < RG; ++k) {
            const int row = row0 + k;
            const bool vis = (row < a.R) && (key < x.t1) && (key <= lim + row / a.G);
            if (!vis) v[k] = -INFINITY;
          }
        }
      };
      // v becomes x = S*c - m_ref (log2 units)
      auto to_log2 = [&](float (&v)[RG]) {
#pragma unroll
        for (int k = 0; k < RG; k += 4) {
          const float4 m = *reinterpret_cast<const float4*>(&M.mref[row0 + k]);
          v[k] = fmaf(v[k], c_log2, -m.x);
          v[k + 1] = fmaf(v[k + 1], c_log2, -m.y);
          v[k + 2] = fmaf(v[k + 2], c_log2, -m.z);
          v[k + 3] = fmaf(v[k + 3], c_log2, -m.w);
        }
      };
      // the item's first tile sets every row's reference max (it starts at
      // kNoMax), so it skips the check: v keeps the raw scores for the max
      float v[RG];
      load_scores(v);
      bool ex = jl == 0;
      if (jl > 0) {
        to_log2(v);
#pragma unroll
        for (int k = 0; k < RG; ++k) ex |= v[k] > kTau;
      }
      const int f = vote(ex);
      if (f & 2) return;
      if (f & 1) {
        // tile max of the group's rows from the raw scores (reloaded after a check)
        if (jl > 0) load_scores(v);
        float mx[BF::Half];
        BF::template run_from<true>(v, mx, lane);
#pragma unroll
        for (int k = 0; k < CNT; ++k) M.red[i][row0 + rbase + k] = mx[k];
        named_bar_sync(bar_id, 128);
        if (gt < RG) {
          const int row = row0 + gt;
          const float m_old = M.mref[row];
          const float tmax = fmaxf(fmaxf(M.red[0][row], M.red[1][row]), fmaxf(M.red[2][row], M.red[3][row]));
          const float m_new = fmaxf(m_old, tmax * c_log2);  // tmax = -inf keeps m_old
          M.mref[row] = m_new;
          M.alpha[row] = (m_new == m_old) ? 1.0f : exp2f(m_old - m_new);
        }
        named_bar_sync(bar_id, 128);
        bool resc = false;
#pragma unroll
        for (int k = 0; k < RG; k += 4) {
          const float4 al = *reinterpret_cast<const float4*>(&M.alpha[row0 + k]);
          lsum[k] *= al.x, lsum[k + 1] *= al.y, lsum[k + 2] *= al.z, lsum[k + 3] *= al.w;
          resc |= (al.x != 1.0f) | (al.y != 1.0f) | (al.z != 1.0f) | (al.w != 1.0f);
        }
        if (resc && jl > 0) {
          // O^T holds tiles < j of this item: wait for PV(j-1), then scale
          // the group's columns (rows) by alpha
          bad |= !mbar_wait(&M.pv_done[(j - 1) % kPBufs], ((j - 1) / kPBufs) & 1, abort);
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < kHalves; ++h) {
#pragma unroll
            for (int c = 0; c < RG / 8; ++c) {
              uint32_t r[8];
              const uint32_t ta = lane_base + ocol + 64 * h + row0 + 8 * c;
              PA_TMEM_LD_X8(ta, r);
              tmem_wait_ld();
              reg_fence(r);
#pragma unroll
              for (int k = 0; k < 8; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * M.alpha[row0 + 8 * c + k]);
              PA_TMEM_ST_X8(ta, r);
            }
          }
          tmem_wait_st();
        }
        if (jl > 0) load_scores(v);  // reloaded rather than held across the rescale
        to_log2(v);
      }
      // probabilities with the (possibly moved) references -> the P^T row
      // of this key (MN-major: one 128-byte row per key, 8-row pieces
      // swizzled).  A masked score is -inf, so its probability is exactly 0.
#pragma unroll
      for (int c8 = 0; c8 < RG / 8; ++c8) {
        float p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) p[k] = ex2_approx(v[8 * c8 + k]);
        __half2 h0 = __floats2half2_rn(p[0], p[1]);
        __half2 h1 = __floats2half2_rn(p[2], p[3]);
        __half2 h2 = __floats2half2_rn(p[4], p[5]);
        __half2 h3 = __floats2half2_rn(p[6], p[7]);
        uint4 w;
        w.x = *reinterpret_cast<uint32_t*>(&h0);
        w.y = *reinterpret_cast<uint32_t*>(&h1);
        w.z = *reinterpret_cast<uint32_t*>(&h2);
        w.w = *reinterpret_cast<uint32_t*>(&h3);
        const int piece = row0 / 8 + c8;
        *reinterpret_cast<uint4*>(prow + ((piece ^ (gt & 7)) << 4)) = w;
#pragma unroll
        for (int k = 0; k < 8; ++k) lsum[8 * c8 + k] += p[k];
      }
      // P^T buffer pb complete (this group's rows) and any O^T rescale of this
      // tile stored; S[j&1] was read for the last time by this group
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.p_full[pb]);
    }
    // ---- epilogue: (m, l, O) partials of the group's rows of this item
    BF::template run<false>(lsum, lane);
#pragma unroll
    for (int k = 0; k < CNT; ++k) M.red[i][row0 + rbase + k] = lsum[k];
    named_bar_sync(bar_id, 128);
    const size_t pi = panel_index(a, x);
    if (gt < RG && row0 + gt < a.R) {
      const int row = row0 + gt;
      const float l = (M.red[0][row] + M.red[1][row]) + (M.red[2][row] + M.red[3][row]);
      a.panel_ml[pi + row] = make_float2(l > 0.f ? M.mref[row] : -INFINITY, l);
    }
    bad |= !mbar_wait(&M.pv_done[(j - 1) % kPBufs], ((j - 1) / kPBufs) & 1, abort);
    tc_fence_after();
    if constexpr (kHalves * RG <= 48) {
      // the group's O^T columns into registers, O^T released to the next
      // item's PV products, then the stores
      uint32_t r[kHalves][RG];
#pragma unroll
      for (int h = 0; h < kHalves; ++h) tmem_load_rows(lane_base + ocol + 64 * h + row0, r[h]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.o_free[n % OBuf<Fmt>::kBufs]);
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
#pragma unroll
        for (int k = 0; k < RG; ++k) {
          const int row = row0 + k;
          if (row < a.R) st_global_hint(a.panel_o + (pi + row) * Fmt::D + h * 128 + gt, __uint_as_float(r[h][k]), keep);
        }
      }
    } else {
      // 64 packed rows of D 256: one half at a time (register budget)
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        uint32_t r[RG];
        tmem_load_rows(lane_base + ocol + 64 * h + row0, r);
#pragma unroll
        for (int k = 0; k < RG; ++k) {
          const int row = row0 + k;
          if (row < a.R) st_global_hint(a.panel_o + (pi + row) * Fmt::D + h * 128 + gt, __uint_as_float(r[k]), keep);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.o_free[n % OBuf<Fmt>::kBufs]);
    }
    named_bar_sync(bar_id, 128);  // every warp of the group is done with mref and red
    // the group's partials of this item are stored: one more arrival for the
    // request (a release, cumulative over the group's stores before the barrier)
    if (gt == 0) red_release_add_u32(a.arrive + x.b, 1u);
    if (gt < RG) M.mref[row0 + gt] = kNoMax;
    named_bar_sync(bar_id, 128);
  }
}

// Merge phase (after the CTA's own items): log-sum-exp combine of the split
// partials into the output rows ("perf(fa2): port decode GQA group-swap into
// d128 varlen launcher", vllm.cpp pull request #48: with num_splits > 1 the
// split partials are merged by their log-sum-exp).  For one output row
// (request b, KV head g, packed row r = qi * G + hl) with splits s = 0 .. S-1:
//   M = max_s m_s,  w_s = 2^(m_s - M),  out = scale * sum_s w_s O_s / sum_s w_s l_s
// with m in log2 units, the sum over s in ascending order and the weights'
// sum by a fixed reduction tree, so the bits depend on S alone (batch
// invariance).  A row with no visible key (M = -inf), a request of length 0
// and a request flagged by an input check write +0.0.
// A task is 128 consecutive elements d of one row (one thread per d); tasks
// run over the rows of every (request, KV head) in schedule order and are
// handed out by a counter in the workspace to five workers of 128 threads per
// CTA.  A task waits, bounded, until every split item of its request has
// arrived (two softmax groups per item); each CTA's items are done before it
// takes a task, and the launch is cooperative, so every item is being worked
// on by a resident CTA.
constexpr int kMergeWorkers = kThreads / 128;
static_assert(kMergeWorkers <= 5 && kMaxSplits <= 64, "merge worker state and weight layout");

template <class Fmt>
__device__ __forceinline__ void merge_phase(const SplitArgs& a, Misc& M, int tid) {
  constexpr int kHalves = Fmt::D / 128;
  const int w = tid >> 7;
  const int e = tid & 127;
  const int bar = 3 + w;  // named barriers 3 .. 3 + kMergeWorkers - 1
  const int per_req = a.Hkv * a.R * kHalves;
  const int total = a.B * per_req;
  const float scale = Fmt::kElemBytes == 1 ? __ldg(a.v_scale) : 1.0f;
  while (true) {
    if (e == 0) M.ctask[w] = atomicAdd(a.queue, 1u);
    named_bar_sync(bar, 128);
    const int t = M.ctask[w];
    if (t >= total) break;
    const int b = M.sched.order[t / per_req];
    const int rr = (t % per_req) / kHalves;  // row of the request (KV head major)
    const int g = rr / a.R, row = rr % a.R;
    const int d = (t % kHalves) * 128 + e;
    int ns = M.sched.nsplit[b];
    if (e == 0) {
      const uint32_t want = 2u * (uint32_t)ns * (uint32_t)a.Hkv;
      const long long t0 = clock64();
      int ok = 1;
      while (ld_acquire_u32(a.arrive + b) < want) {
        if (clock64() - t0 > M.ctl.limit) {
          ok = 0;
          break;
        }
      }
      M.cok[w] = ok;
    }
    named_bar_sync(bar, 128);
    if (!M.cok[w]) {
      if (e == 0) atomicOr(a.status, 0x4u);
      break;
    }
    if (__ldcg(a.bad + b) != 0u) ns = 0;
    const int qi = row / a.G, hl = row % a.G;
    const size_t orow = (size_t)(b * a.q_len + qi) * a.Hq + g * a.G + hl;
    const size_t prow = (size_t)(b * a.Hkv + g) * a.s_max * a.R + row;  // panel row of split 0; split s at + s * R
    // the partial O of every split into the worker's area of the (now idle)
    // pipeline shared memory, requested before the weights are known so that
    // the two rounds of loads overlap; element (s, e) at stage[s * 128 + e]
    const float* o0 = a.panel_o + prow * Fmt::D + d;
    const size_t sstride = (size_t)a.R * Fmt::D;
    const uint32_t stage = smem_u32(smem_base()) + (uint32_t)(w * kMaxSplits * 128 + e) * 4u;
    for (int s = 0; s < ns; ++s) cp_async_4(stage + (uint32_t)s * 512u, o0 + s * sstride);
    // one warp, splits s and s + 32 on lane s: M = max_s m_s, w_s = 2^(m_s - M),
    // lsum = sum_s w_s l_s (a fixed reduction tree, so the bits depend on ns only)
    if (e < 32) {
      const int s = e;
      float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
      if (s < ns) {
        const float2 ml = __ldcg(a.panel_ml + prow + (size_t)s * a.R);
        m0 = ml.x, l0 = ml.y;
      }
      if (s + 32 < ns) {
        const float2 ml = __ldcg(a.panel_ml + prow + (size_t)(s + 32) * a.R);
        m1 = ml.x, l1 = ml.y;
      }
      float Mx = fmaxf(m0, m1);
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, k));
      const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - Mx);
      const float w1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - Mx);
      float ls = w0 * l0 + w1 * l1;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, k);
      if (s < kMaxSplits) M.cw[w][s] = w0;
      if (s + 32 < kMaxSplits) M.cw[w][s + 32] = w1;
      if (s == 0) {
        M.clsum[w] = ls;
        if (a.lse != nullptr && d == 0)
          a.lse[orow] = (Mx == -INFINITY || !(ls > 0.f)) ? -INFINITY : (Mx + log2f(ls)) * 0.6931471805599453f;
      }
    }
    named_bar_sync(bar, 128);
    cp_async_wait_all();  // this thread's own partials (it reads no other thread's)
    const float lsum = M.clsum[w];
    float val = 0.f;
    if (lsum > 0.f) {
      // accumulation in ascending split order
      const float* so = reinterpret_cast<const float*>(smem_base()) + w * kMaxSplits * 128 + e;
      float acc = 0.f;
      for (int s = 0; s < ns; ++s) acc = fmaf(M.cw[w][s], so[s * 128], acc);
      val = acc / lsum * scale;
    }
    if constexpr (Fmt::kQBf16) {
      reinterpret_cast<__nv_bfloat16*>(a.out)[orow * Fmt::D + d] = __float2bfloat16_rn(val);
    } else {
      reinterpret_cast<__half*>(a.out)[orow * Fmt::D + d] = __float2half_rn(val);
    }
    named_bar_sync(bar, 128);  // the worker's weights are read before the next task overwrites them
  }
}

template <class Fmt, int NM, int TMA>
__global__ void __launch_bounds__(kThreads, 1) split_kernel(const __grid_constant__ SplitArgs a) {
  using L = Layout<Fmt, NM>;
  uint8_t* sm = smem_base();
  Misc& M = *reinterpret_cast<Misc*>(sm + L::kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the request lengths and the block table are the first things the
  // schedule and the loaders read: their loads start before the prologue
  const int len_t = tid < a.B ? ld_page_id(a.ctx_lens + tid) : 0;
  if (warp == 2) {
    const size_t bt_bytes = (size_t)a.B * a.mpr * 4;
    const size_t n = bt_bytes < 65536 ? bt_bytes : 65536;
    for (size_t off = (size_t)lane * 128; off < n; off += 32 * 128)
      prefetch_l2(reinterpret_cast<const char*>(a.block_table) + off);
  }

  if (tid == 0) {
    mbar_init(&M.kst_full, TMA != 0 ? 1 : 32);
    mbar_init(&M.vst_full, TMA != 0 ? 1 : 32);
    mbar_init(&M.kst_empty, 4);
    mbar_init(&M.vst_empty, 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&M.kbuf_full[s], 4);
      mbar_init(&M.s_full[s], 1);
      mbar_init(&M.vtile_full[s], 4);
    }
    for (int s = 0; s < kPBufs; ++s) {
      mbar_init(&M.p_full[s], 8);  // the eight softmax warps
      mbar_init(&M.pv_done[s], 1);
    }
    mbar_init(&M.q_full, 1);
    mbar_init(&M.q_empty, 1);
    mbar_init(&M.o_free[0], 8);
    mbar_init(&M.o_free[1], 8);
    mbar_init(&M.fin, 1);
    mbar_init(&M.fin_qk, 1);
    M.ctl.abort = 0;
    M.ctl.limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimitCycles;
    for (int w = 0; w < 16; ++w) M.vote[w / 8][(w / 4) & 1][w % 4] = 0;
    mbar_fence_init();
  }
  if (tid < kMaxRows) M.mref[tid] = kNoMax;
  if (warp == 1) tmem_alloc(&M.tmem_base, 512);
  // zero the Q tile (rows >= R stay zero) and both P^T buffers (rows >= N stay zero)
  for (int o = tid * 16; o < L::kQBytes; o += kThreads * 16)
    *reinterpret_cast<uint4*>(sm + L::kOffQ + o) = make_uint4(0, 0, 0, 0);
  for (int o = tid * 16; o < kPBufs * 16384; o += kThreads * 16)
    *reinterpret_cast<uint4*>(sm + L::kOffP + o) = make_uint4(0, 0, 0, 0);
  sched_build(M.sched, len_t, a.B, a.Hkv, a.max_ctx, a.status, a.bad);  // contains __syncthreads
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = M.tmem_base;

  // warp w runs on sub-partition w % 4; the TMEM lane quarter of the K decode
  // and softmax warps is w % 4 as well.  The V decode warps, the heaviest
  // users of the shared-memory queues, sit on sub-partitions 0 and 2, away
  // from the PV issuer (sub-partition 1) and the QK issuer (sub-partition 3).
  const int vq = warp == 0 ? 0 : warp == 8 ? 1 : warp == 2 ? 2 : warp == 10 ? 3 : -1;
  if (warp == 3 || warp == 9) {
    const bool is_v = warp == 9;
    // TMA: 1 = one thread (pages of a tile or more), 2 = the warp (shorter
    // pages), 3 = one thread, 272-byte windows (bases 8 bytes past a 16-byte
    // boundary); a separate instantiation each, so no kernel carries two
    if constexpr (TMA == 2) {
      role_loader_tma_blocks<Fmt>(a, M, is_v, sm + (is_v ? L::kOffVst : L::kOffKst), lane);
    } else if constexpr (TMA == 1 || TMA == 3) {
      if (lane == 0) role_loader_tma<Fmt, TMA == 3>(a, M, is_v, sm + (is_v ? L::kOffVst : L::kOffKst));
    } else {
      role_loader_cp<Fmt>(a, M, is_v, lane, sm + (is_v ? L::kOffVst : L::kOffKst));
    }
    __syncwarp();
  } else if (warp == 11) {
    role_q_qk<Fmt, NM>(a, M, lane, sm + L::kOffQ, tb);
    if (lane == 0) {
      mma_commit(&M.fin_qk);  // the same drain for the QK products
      const long long t0 = clock64();
      while (!mbar_try_wait(&M.fin_qk, 0) && clock64() - t0 < M.ctl.limit) {
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      role_pv<Fmt, NM>(a, M, tb, smem_u32(sm + L::kOffP), smem_u32(sm + L::kOffV));
      // drain: every PV this thread issued must finish before TMEM is released
      mma_commit(&M.fin);
      const long long t0 = clock64();
      while (!mbar_try_wait(&M.fin, 0) && clock64() - t0 < M.ctl.limit) {
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    role_kdecode<Fmt, TMA == 3>(a, M, warp - 4, lane, tb, sm + L::kOffKst);
  } else if (vq >= 0) {
    role_vdecode<Fmt, NM, TMA == 3>(a, M, vq, lane, sm + L::kOffVst, sm + L::kOffV);
  } else {
    role_softmax<Fmt, NM>(a, M, (warp - 12) / 4, warp & 3, lane, tb, sm + L::kOffP);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
  if (M.ctl.abort) {
    if (tid == 0) atomicOr(a.status, 0x4u);  // the call's output is invalid; other CTAs' merge waits run out
  } else {
    merge_phase<Fmt>(a, M, tid);
  }
  // the last CTA to finish returns the per-call words of the workspace to
  // zero for the next call (every CTA has finished reading them by then)
  __syncthreads();
  if (tid == 0 && atom_add_acq_rel_u32(a.done, 1u) == gridDim.x - 1) {
    for (int b = 0; b < a.B; ++b) a.arrive[b] = 0u, a.bad[b] = 0u;
    *a.queue = 0u;
    *a.done = 0u;
  }
}

template <class Fmt, int NM, int TMA>
cudaError_t launch_one(const SplitArgs& a, int grid, cudaStream_t stream) {
  constexpr int kSmem = Layout<Fmt, NM>::kSmemBytes;
  auto kern = split_kernel<Fmt, NM, TMA>;
  // the attribute is per device; setting it is idempotent, so a racing second
  // setter is harmless
  static std::atomic<uint64_t> set_on_devices{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(set_on_devices.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    set_on_devices.fetch_or(bit);
  }
  // cooperative: the merge phase waits for split items of other CTAs, so
  // every CTA of the grid must be resident at once (one per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class Fmt, int TMA>
cudaError_t launch_mode(const SplitArgs& a, int grid, cudaStream_t stream) {
  switch ((a.R + 15) / 16 * 16) {
    case 16: return launch_one<Fmt, 16, TMA>(a, grid, stream);
    case 32: return launch_one<Fmt, 32, TMA>(a, grid, stream);
    case 48: return launch_one<Fmt, 48, TMA>(a, grid, stream);
    case 64: return launch_one<Fmt, 64, TMA>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// One element format's launcher (each format's instantiations live in their
// own translation unit, split_kv_<format>.cu, so they compile in parallel).
#define PA_DEFINE_SPLIT_LAUNCHER(name, Fmt)                                          \
  cudaError_t name(const SplitArgs& a, int grid, cudaStream_t stream) {              \
    if (a.kv_load == kKvLoadCopy) return launch_mode<Fmt, 0>(a, grid, stream);       \
    if (a.kv_load == kKvLoadWindow) return launch_mode<Fmt, 3>(a, grid, stream);     \
    return a.page_size < kTileKeys ? launch_mode<Fmt, 2>(a, grid, stream)            \
                                   : launch_mode<Fmt, 1>(a, grid, stream);           \
  }

}  // namespace pa
