// Split-KV paged decode / speculative-verify attention on the sm_103a tensor
// cores (tcgen05 + TMEM), for two element formats:
//   Fp8Fmt : FP16 Q, E4M3 K/V with FP32 per-tensor scales, head_dim 256
//   Bf16Fmt: BF16 Q/K/V, head_dim 128
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
// accumulation for both QK and PV).  For E4M3, K' and V' are the codes decoded
// exactly to FP16; for BF16, K' is K and V' is V converted to FP16 so
// that P can stay FP16 in the PV product.  Each TMEM lane is one key, so the
// online softmax of a row is a reduction across lanes (warp shuffles).
//
// Warp roles (16 warps):
//   0  K loader   TMA (or cp.async for 8-byte aligned data) of block-table-
//                 gathered K rows into a 32-key staging ring
//   2  V loader   the same for V
//   3  Q loader   the packed Q tile of each item (128-byte swizzle)
//   1  MMA        one thread issues tcgen05.mma and commits to mbarriers
//   4-7  K decode staging -> K' in TMEM (lane = key), the QK A operand
//   8-11 V decode staging -> V' in the MN-major SMEM operand
//   12-15 softmax masking, lazy-max online softmax, P^T, row sums, O^T rescale,
//         and the item's FP32 (m, l, O) partials written to the workspace.
// Every wait is bounded (see mbar_wait); a wait that runs out aborts the CTA
// cleanly, frees TMEM and raises PA_FLAG_TIMEOUT.
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
  static constexpr int kQBf16 = 0;                 // Q (and K') type of the QK product
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

struct Bf16Fmt {
  static constexpr int D = 128;
  static constexpr int kElemBytes = 2;
  static constexpr int kQBf16 = 1;
  static __device__ __forceinline__ float score_scale(const float*) {
    return 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
  }
  // BF16x2 word -> FP16x2 word (exact for |x| in [2^-14, 65504]; smaller
  // magnitudes round to the FP16 subnormal grid)
  static __device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

constexpr int kStages = 4;         // staging ring depth per tensor, in 32-key chunks
constexpr int kChunkKeys = 32;
constexpr int kPageSeg = 8;       // chunks whose page ids a loader lane holds in registers
constexpr float kTau = 8.0f;       // a row's reference max moves only when a score exceeds it by 2^8
constexpr float kNoMax = -1e30f;   // reference max of a row that has seen no key (finite: 2^(s - kNoMax) never NaN)
constexpr int kThreads = 512;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                         // up to 4 atoms x 64 rows x 128 B
constexpr int kOffV = 32768;                     // up to 4 atoms x 128 keys x 128 B
constexpr int kOffP = kOffV + 65536;             // 2 x (128 keys x 128 B)
constexpr int kOffKst = kOffP + 2 * 16384;       // kStages x 32 keys x 256 B
constexpr int kOffVst = kOffKst + kStages * 8192;
constexpr int kOffMisc = kOffVst + kStages * 8192;

// TMEM column map (512 columns allocated)
constexpr uint32_t kColS = 0;     // S^T, 2 buffers of 64 columns
constexpr uint32_t kColO = 128;   // O^T, d 0..127 at +0, d 128..255 at +64
constexpr uint32_t kColK = 256;   // K' operand, 2 buffers of 128 columns

struct Misc {
  uint64_t kst_full[kStages], kst_empty[kStages], vst_full[kStages], vst_empty[kStages];
  uint64_t kbuf_full[2], kbuf_empty[2], s_full[2], s_empty[2], p_full[2], pv_done[2];
  uint64_t vbuf_full, q_full, q_empty, o_free, grp, fin;
  uint32_t tmem_base;
  WaitCtl ctl;
  int exceed_tag[2][4];
  int rescale_tag;
  alignas(16) float mref[kMaxRows];  // read as float4
  alignas(16) float thr[kMaxRows];   // (mref + tau) / c: scores above this need a new reference
  alignas(16) float alpha[kMaxRows];
  alignas(16) float red[4][kMaxRows];
  Sched sched;
};
static_assert(offsetof(Misc, mref) % 16 == 0, "mref is read with 16-byte loads");
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc) + 1024;

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

// ------------------------------------------------------------------ roles --

// Key row kk of a stage (see role_loader) as 16 pieces of 16 bytes; zeros
// for keys past the split end (their stage bytes are stale or a page tail).
__device__ __forceinline__ void load_stage_row(const uint8_t* stage, int kk, bool live, uint4 (&raw)[16]) {
#pragma unroll
  for (int p = 0; p < 16; ++p)
    raw[p] = live ? *reinterpret_cast<const uint4*>(stage + (p >> 3) * 4096 + kk * 128 + (((p & 7) ^ (kk & 7)) << 4))
                  : make_uint4(0u, 0u, 0u, 0u);
}

// K or V loader: 32-key chunks into the staging ring.  Chunk c of the CTA's
// item sequence goes to stage c % kStages.  Stage layout: two halves of the
// 256-byte key rows, half h at h*4096, key kk's 128 bytes at kk*128 with its
// 16-byte piece p at ((p ^ (kk & 7)) * 16) (the TMA 128-byte swizzle), so the
// decode warps read eight consecutive keys without bank conflicts.
//
// TMA mode (16-byte aligned bases and strides): one thread issues, per 16-key
// block, two 2 KB boxes (row bytes 0-127 and 128-255) of the 4-D byte view
// (row byte, KV head, slot, page); completion is counted in bytes on the
// stage's full barrier.  Blocks entirely past the split end are not loaded.
// cp.async mode (8-byte aligned data): every lane copies 8-byte pieces of the
// chunk's rows into the same layout, zero-filling rows past the split end.
template <int USE_TMA>
__device__ __forceinline__ void role_loader(const SplitArgs& a, Misc& M, bool is_v, int lane) {
  const uint8_t* base = is_v ? a.v : a.k;
  const long long pstr = is_v ? a.v_ps : a.k_ps;
  const long long tstr = is_v ? a.v_ts : a.k_ts;
  const long long hstr = is_v ? a.v_hs : a.k_hs;
  const CUtensorMap* map = is_v ? &a.v_map : &a.k_map;
  uint64_t* full = is_v ? M.vst_full : M.kst_full;
  uint64_t* empty = is_v ? M.vst_empty : M.kst_empty;
  uint8_t* ring = smem_base() + (is_v ? kOffVst : kOffKst);
  WaitCtl* abort = &M.ctl;
  uint32_t c = 0;
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int32_t* bt = a.block_table + (size_t)x.b * a.mpr;
    const uint8_t* hbase = base + (long long)x.g * hstr;
    const int nchunks = tiles_of(x) * (kTileKeys / kChunkKeys);
    // Page id of key t0 + 32*cj + lane, for 8 chunks at a time in registers:
    // `cur` serves chunks cs..cs+7 while `nxt` is being loaded for cs+8..cs+15,
    // so the block-table latency (long under full HBM load) stays hidden.
    auto load_segment = [&](int (&pg)[kPageSeg], int cs) {
#pragma unroll
      for (int s = 0; s < kPageSeg; ++s) {
        const int cj = cs + s;
        const int t = x.t0 + cj * kChunkKeys + lane;
        pg[s] = (cj < nchunks && t < x.t1) ? __ldg(bt + t / a.page_size) : -1;
      }
    };
    int cur[kPageSeg], nxt[kPageSeg];
    load_segment(cur, 0);
    load_segment(nxt, kPageSeg);
    for (int cs = 0; cs < nchunks; cs += kPageSeg) {
#pragma unroll
      for (int s = 0; s < kPageSeg; ++s) {
        const int ci = cs + s;
        if (ci >= nchunks) break;
        const int st = c % kStages;
        const uint32_t ph = (c / kStages) & 1;
        const int page_cur = cur[s];
        if (!mbar_wait(&empty[st], ph ^ 1, abort)) goto done;
        const int kb = x.t0 + ci * kChunkKeys;
        const uint32_t dst0 = smem_u32(ring + st * (kChunkKeys * 256));
        if constexpr (USE_TMA) {
          // lanes 0 and 16 hold the pages of the chunk's two 16-key blocks
          const int t = kb + lane;
          bool ok = (lane & 15) == 0 && t < x.t1;
          if (ok && (unsigned)page_cur >= (unsigned)a.num_pages) {
            atomicOr(a.status, 0x1u);
            atomicOr(a.bad + x.b, 1u);
            ok = false;
          }
          const unsigned okmask = __ballot_sync(0xffffffffu, ok);
          const int pg0 = __shfl_sync(0xffffffffu, page_cur, 0), pg1 = __shfl_sync(0xffffffffu, page_cur, 16);
          if (lane == 0) {
            const uint32_t blocks = (okmask & 1u) + ((okmask >> 16) & 1u);
            mbar_arrive_expect_tx(&full[st], 4096u * blocks);
#pragma unroll
            for (int sb = 0; sb < 2; ++sb) {
              if (!(okmask >> (16 * sb) & 1u)) continue;
              const int pg = sb ? pg1 : pg0;
              const int slot = (kb + 16 * sb) % a.page_size;
              tma_load_4d(dst0 + sb * 2048, map, 0, x.g, slot, pg, &full[st]);
              tma_load_4d(dst0 + 4096 + sb * 2048, map, 128, x.g, slot, pg, &full[st]);
            }
          }
          __syncwarp();
        } else {
          const int t = kb + lane;
          long long rowoff = -1;
          if (t < x.t1) {
            if ((unsigned)page_cur < (unsigned)a.num_pages) {
              rowoff = (long long)page_cur * pstr + (long long)(t % a.page_size) * tstr;
            } else {
              atomicOr(a.status, 0x1u);
              atomicOr(a.bad + x.b, 1u);
            }
          }
#pragma unroll 4
          for (int kk = 0; kk < kChunkKeys; ++kk) {
            const long long ro = __shfl_sync(0xffffffffu, rowoff, kk);
            const int piece = lane >> 1;  // 16-byte piece 0..15 of the row
            const uint8_t* src = ro >= 0 ? hbase + ro + lane * 8 : base;
            const uint32_t dst =
                dst0 + (piece >> 3) * 4096 + kk * 128 + (((piece & 7) ^ (kk & 7)) << 4) + (lane & 1) * 8;
            cp_async_8(dst, src, ro >= 0 ? 8u : 0u);
          }
          cp_async_arrive(&full[st]);
        }
        ++c;
      }
#pragma unroll
      for (int s = 0; s < kPageSeg; ++s) cur[s] = nxt[s];
      load_segment(nxt, cs + 2 * kPageSeg);
    }
  }
done:
  if constexpr (!USE_TMA) cp_async_wait_all();
}

// Q loader: packed row r = qi * G + hl holds query head g*G + hl of verify
// query qi.  K-major operand: element (r, d) at (d/64)*8192 + r*128 +
// ((((d%64)/8) ^ (r%8)) * 16) + (d%8)*2.
template <class Fmt>
__device__ __forceinline__ void role_qload(const SplitArgs& a, Misc& M, int lane) {
  constexpr int kPieces = Fmt::D / 8;  // 16-byte pieces per Q row
  uint8_t* qbuf = smem_base() + kOffQ;
  WaitCtl* abort = &M.ctl;
  const uint16_t* q = reinterpret_cast<const uint16_t*>(a.q);
  uint32_t n = 0;
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x, ++n) {
    const Item x = sched_item(M.sched, a.B, it);
    if (!mbar_wait(&M.q_empty, (n & 1) ^ 1, abort)) break;
    for (int u = lane; u < a.R * kPieces; u += 32) {
      const int r = u / kPieces, c = u % kPieces;  // piece c holds d = 8c .. 8c+7
      const int qi = r / a.G, hl = r % a.G;
      const uint16_t* src = q + ((size_t)(x.b * a.q_len + qi) * a.Hq + x.g * a.G + hl) * Fmt::D + c * 8;
      const uint32_t dst = smem_u32(qbuf + (c >> 3) * 8192 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
      cp_async_16(dst, src, 16u);
    }
    // the tensor core reads Q through the async proxy: land the copies, fence,
    // then signal
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && !a.withhold_q) mbar_arrive(&M.q_full);  // withheld only by the timeout test hook
  }
  cp_async_wait_all();
}

// K decode: warp quarter i owns TMEM lanes 32i..32i+31 = keys 32i.. of each
// tile; lane = key, column c holds elements d = 2c, 2c+1.
template <class Fmt>
__device__ __forceinline__ void role_kdecode(const SplitArgs& a, Misc& M, int i, int lane, uint32_t tb) {
  uint8_t* ring = smem_base() + kOffKst;
  WaitCtl* abort = &M.ctl;
  uint32_t j = 0;
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    for (int jl = 0; jl < nt; ++jl, ++j) {
      const uint32_t c = 4 * j + i;
      const int st = c % kStages;
      if (!mbar_wait(&M.kst_full[st], (c / kStages) & 1, abort)) return;
      // take this key's 256-byte row into registers and hand the stage back
      // at once, so the loader's refill does not wait for the tensor core
      uint4 raw[16];
      load_stage_row(ring + st * (kChunkKeys * 256), lane, x.t0 + jl * kTileKeys + 32 * i + lane < x.t1, raw);
      mbar_arrive(&M.kst_empty[st]);
      if (!mbar_wait(&M.kbuf_empty[j & 1], ((j >> 1) & 1) ^ 1, abort)) return;
      const uint32_t taddr = tb + ((uint32_t)(32 * i) << 16) + kColK + (j & 1) * 128;
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
          for (int h = 0; h < 4; ++h) {
            const uint4 w = raw[4 * c4 + h];
            r[4 * h + 0] = w.x, r[4 * h + 1] = w.y, r[4 * h + 2] = w.z, r[4 * h + 3] = w.w;
          }
          PA_TMEM_ST_X16(taddr + c4 * 16, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.kbuf_full[j & 1]);
    }
  }
}

// V decode: keys 32i.. of each tile into the MN-major V' operand: element
// (key, d) at (d/64)*16384 + key*128 + ((((d%64)/8) ^ (key%8)) * 16) + (d%8)*2.
template <class Fmt>
__device__ __forceinline__ void role_vdecode(const SplitArgs& a, Misc& M, int i, int lane) {
  uint8_t* sm = smem_base();
  uint8_t* ring = sm + kOffVst;
  uint8_t* vbuf = sm + kOffV;
  WaitCtl* abort = &M.ctl;
  uint32_t j = 0;
  const int key = 32 * i + lane;
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    for (int jl = 0; jl < nt; ++jl, ++j) {
      const uint32_t c = 4 * j + i;
      const int st = c % kStages;
      if (!mbar_wait(&M.vst_full[st], (c / kStages) & 1, abort)) return;
      // row into registers, stage back to the loader, then wait for PV(j-1)
      uint4 raw[16];
      load_stage_row(ring + st * (kChunkKeys * 256), lane, x.t0 + jl * kTileKeys + key < x.t1, raw);
      mbar_arrive(&M.vst_empty[st]);
      if (j > 0 && !mbar_wait(&M.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort)) return;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 x4 = raw[ch];
        if constexpr (Fmt::kElemBytes == 1) {
          // piece ch = d 16ch .. 16ch+15 -> two 8-element FP16 pieces
          uint32_t w[8];
          Fmt::decode16(x4, w);
          const int at = ch >> 2, u = ch & 3;
          uint8_t* dst = vbuf + at * 16384 + key * 128;
          *reinterpret_cast<uint4*>(dst + (((2 * u) ^ (key & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + (((2 * u + 1) ^ (key & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          // piece ch = d 8ch .. 8ch+7
          const uint4 h = make_uint4(Fmt::bf2_to_h2(x4.x), Fmt::bf2_to_h2(x4.y), Fmt::bf2_to_h2(x4.z),
                                     Fmt::bf2_to_h2(x4.w));
          const int at = ch >> 3, u = ch & 7;
          *reinterpret_cast<uint4*>(vbuf + at * 16384 + key * 128 + ((u ^ (key & 7)) << 4)) = h;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.vbuf_full);
    }
  }
}

// MMA issuer (one thread).  QK of tile j is issued before PV of tile j-1 so
// the tensor core computes the next scores while the softmax warps work.
template <class Fmt, int NM>
__device__ __forceinline__ void role_mma(const SplitArgs& a, Misc& M, uint32_t tb) {
  uint8_t* sm = smem_base();
  const uint32_t qbase = smem_u32(sm + kOffQ);
  const uint32_t vbase = smem_u32(sm + kOffV);
  const uint32_t pbase = smem_u32(sm + kOffP);
  constexpr uint32_t id_qk = idesc_f16(128, NM, Fmt::kQBf16, 0, 0);
  constexpr uint32_t id_pv = idesc_f16(128, NM, 0, 1, 1);
  constexpr int kKSteps = Fmt::D / 16;
  constexpr int kHalves = Fmt::D / 128;
  WaitCtl* abort = &M.ctl;
  uint32_t j = 0, n = 0;
  bool ok = true;
  auto issue_pv = [&](uint32_t jj, bool first) -> bool {
    if (!mbar_wait(&M.p_full[jj & 1], (jj >> 1) & 1, abort)) return false;
    if (!mbar_wait(&M.vbuf_full, jj & 1, abort)) return false;
    if (first && !mbar_wait(&M.o_free, (n & 1) ^ 1, abort)) return false;
    tc_fence_after();
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = sdesc_sw128(vbase + 2 * h * 16384 + kk * 2048, 16384, 1024);
        const uint64_t bd = sdesc_sw128(pbase + (jj & 1) * 16384 + kk * 2048, 16384, 1024);
        mma_ss(tb + kColO + 64 * h, ad, bd, id_pv, (first && kk == 0) ? 0u : 1u);
      }
    }
    mma_commit(&M.pv_done[jj & 1]);
    return true;
  };
  for (int it = blockIdx.x; ok && it < M.sched.total; it += gridDim.x, ++n) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    if (!mbar_wait(&M.q_full, n & 1, abort)) break;
    for (int jl = 0; jl < nt; ++jl, ++j) {
      if (!mbar_wait(&M.kbuf_full[j & 1], (j >> 1) & 1, abort) ||
          !mbar_wait(&M.s_empty[j & 1], ((j >> 1) & 1) ^ 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        const uint64_t bd = sdesc_sw128(qbase + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
        mma_ts(tb + kColS + (j & 1) * 64, tb + kColK + (j & 1) * 128 + kk * 8, bd, id_qk, kk > 0 ? 1u : 0u);
      }
      mma_commit(&M.s_full[j & 1]);
      mma_commit(&M.kbuf_empty[j & 1]);
      if (jl == nt - 1) mma_commit(&M.q_empty);
      if (jl > 0 && !issue_pv(j - 1, jl == 1)) {
        ok = false;
        break;
      }
    }
    if (ok && !issue_pv(j - 1, nt == 1)) ok = false;
  }
}

// Softmax warps: quarter i reads TMEM lanes 32i.. (keys of S^T, then d of O^T).
//
// Scores stay in S units (the raw QK^T accumulator); c = log2(e) * scale turns
// them into the log2 domain inside one FFMA.  Per row r the group keeps a
// reference max m_r (log2 units; kNoMax before any visible key) and the
// threshold thr_r = (m_r + tau) / c: a tile needs a new reference only if some
// visible score exceeds thr_r, so the common tile is P = 2^(S*c - m_r) with no
// cross-lane reduction.  Each thread keeps the running row sums of its own key
// slot for all rows and the group reduces them once per item.
template <class Fmt, int NM>
__device__ __forceinline__ void role_softmax(const SplitArgs& a, Misc& M, int i, int lane, uint32_t tb) {
  using BF = Butterfly<NM, 16>;
  constexpr int CNT = BF::Count;
  constexpr int kHalves = Fmt::D / 128;
  uint8_t* pbuf = smem_base() + kOffP;
  WaitCtl* abort = &M.ctl;
  const int gt = 32 * i + lane;  // thread index inside the softmax group
  const float c_log2 = Fmt::score_scale(a.k_scale);
  const uint32_t lane_base = tb + ((uint32_t)(32 * i) << 16);
  const int rbase = BF::base(lane);  // rows rbase .. rbase+CNT-1 of every butterfly result
  uint32_t j = 0, gph = 0;
  auto group_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.grp);
    const bool r = mbar_wait(&M.grp, gph, abort);
    gph ^= 1;
    return r;
  };
  for (int it = blockIdx.x; it < M.sched.total; it += gridDim.x) {
    const Item x = sched_item(M.sched, a.B, it);
    const int nt = tiles_of(x);
    const int lim = x.L - a.q_len;  // packed row r sees key t iff t <= lim + r / G
    float lsum[NM];                 // running row sums of this thread's key slot
#pragma unroll
    for (int r = 0; r < NM; ++r) lsum[r] = 0.f;
    for (int jl = 0; jl < nt; ++jl, ++j) {
      if (!mbar_wait(&M.s_full[j & 1], (j >> 1) & 1, abort)) return;
      tc_fence_after();
      const uint32_t s_addr = lane_base + kColS + (j & 1) * 64;
      const int tile0 = x.t0 + jl * kTileKeys;
      const int key = tile0 + gt;
      const int vis_end = min(x.t1, lim + 1);  // keys below this are visible to every row
      const bool masked_tile = tile0 + kTileKeys > vis_end || NM > a.R;
      // 16 scores of columns 16*c16.. from TMEM, masked to -inf where invisible
      auto load_chunk = [&](int c16, float (&v)[16]) {
        uint32_t r[16];
        tmem_load16(s_addr + 16 * c16, r);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
        if (masked_tile) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int row = 16 * c16 + k;
            const bool vis = (row < a.R) && (key < x.t1) && (key <= lim + row / a.G);
            if (!vis) v[k] = -INFINITY;
          }
        }
      };
      // pass 1: does any visible score exceed its row's threshold?
      bool ex = false;
#pragma unroll
      for (int c16 = 0; c16 < NM / 16; ++c16) {
        float v[16];
        load_chunk(c16, v);
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
          const float4 th = *reinterpret_cast<const float4*>(&M.thr[16 * c16 + k]);
          ex |= (v[k] > th.x) | (v[k + 1] > th.y) | (v[k + 2] > th.z) | (v[k + 3] > th.w);
        }
      }
      if (__any_sync(0xffffffffu, ex) && lane == 0) M.exceed_tag[j & 1][i] = (int)j + 1;
      if (!group_sync()) return;
      const int* tag = M.exceed_tag[j & 1];
      const bool slow = tag[0] == (int)j + 1 || tag[1] == (int)j + 1 || tag[2] == (int)j + 1 || tag[3] == (int)j + 1;
      if (slow) {
        // tile max per row: a 16-row butterfly per chunk leaves one row per lane
        using BF16 = Butterfly<16, 16>;
#pragma unroll
        for (int c16 = 0; c16 < NM / 16; ++c16) {
          float v[16], mx[BF16::Half];
          load_chunk(c16, v);
          BF16::template run_from<true>(v, mx, lane);
          M.red[i][16 * c16 + BF16::base(lane)] = mx[0];
        }
        if (!group_sync()) return;
        if (gt < NM) {
          const float m_old = M.mref[gt];
          const float tmax = fmaxf(fmaxf(M.red[0][gt], M.red[1][gt]), fmaxf(M.red[2][gt], M.red[3][gt]));
          const float m_new = fmaxf(m_old, tmax * c_log2);  // tmax = -inf keeps m_old
          const float al = (m_new == m_old) ? 1.0f : exp2f(m_old - m_new);
          M.mref[gt] = m_new;
          M.thr[gt] = (m_new + kTau) / c_log2;
          M.alpha[gt] = al;
          if (al != 1.0f) M.rescale_tag = (int)j + 1;
        }
        if (!group_sync()) return;
        if (M.rescale_tag == (int)j + 1) {
#pragma unroll
          for (int r = 0; r < NM; r += 4) {
            const float4 al = *reinterpret_cast<const float4*>(&M.alpha[r]);
            lsum[r] *= al.x, lsum[r + 1] *= al.y, lsum[r + 2] *= al.z, lsum[r + 3] *= al.w;
          }
          if (jl > 0) {
            // O^T holds tiles < j: wait for PV(j-1), then scale column r by alpha[r]
            if (!mbar_wait(&M.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort)) return;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
#pragma unroll
              for (int c16 = 0; c16 < NM / 16; ++c16) {
                uint32_t r[16];
                const uint32_t ta = lane_base + kColO + 64 * h + 16 * c16;
                tmem_load16(ta, r);
#pragma unroll
                for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * M.alpha[16 * c16 + k]);
                PA_TMEM_ST_X16(ta, r);
              }
            }
            tmem_wait_st();
          }
        }
      }
      // pass 2: probabilities -> P^T row of this key (MN-major: one 128-byte
      // row per key, 8-row pieces swizzled); P[j&1] is free once PV(j-2) is
      // done.  A masked score is -inf, so its probability is exactly 0.
      if (j >= 2 && !mbar_wait(&M.pv_done[j & 1], ((j - 2) >> 1) & 1, abort)) return;
      uint8_t* prow = pbuf + (j & 1) * 16384 + gt * 128;
#pragma unroll
      for (int c16 = 0; c16 < NM / 16; ++c16) {
        float v[16];
        load_chunk(c16, v);
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int c8 = 2 * c16 + h8;
          const float4 m0 = *reinterpret_cast<const float4*>(&M.mref[8 * c8]);
          const float4 m1 = *reinterpret_cast<const float4*>(&M.mref[8 * c8 + 4]);
          const float* u = v + 8 * h8;
          float p[8];
          p[0] = ex2_approx(fmaf(u[0], c_log2, -m0.x));
          p[1] = ex2_approx(fmaf(u[1], c_log2, -m0.y));
          p[2] = ex2_approx(fmaf(u[2], c_log2, -m0.z));
          p[3] = ex2_approx(fmaf(u[3], c_log2, -m0.w));
          p[4] = ex2_approx(fmaf(u[4], c_log2, -m1.x));
          p[5] = ex2_approx(fmaf(u[5], c_log2, -m1.y));
          p[6] = ex2_approx(fmaf(u[6], c_log2, -m1.z));
          p[7] = ex2_approx(fmaf(u[7], c_log2, -m1.w));
          __half2 h0 = __floats2half2_rn(p[0], p[1]);
          __half2 h1 = __floats2half2_rn(p[2], p[3]);
          __half2 h2 = __floats2half2_rn(p[4], p[5]);
          __half2 h3 = __floats2half2_rn(p[6], p[7]);
          uint4 w;
          w.x = *reinterpret_cast<uint32_t*>(&h0);
          w.y = *reinterpret_cast<uint32_t*>(&h1);
          w.z = *reinterpret_cast<uint32_t*>(&h2);
          w.w = *reinterpret_cast<uint32_t*>(&h3);
          *reinterpret_cast<uint4*>(prow + ((c8 ^ (gt & 7)) << 4)) = w;
#pragma unroll
          for (int k = 0; k < 8; ++k) lsum[8 * c8 + k] += p[k];
        }
      }
      // S[j&1] may now be overwritten by QK(j+2)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.s_empty[j & 1]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.p_full[j & 1]);
    }
    // ---- epilogue: (m, l, O) partials of this item
    BF::template run<false>(lsum, lane);
#pragma unroll
    for (int k = 0; k < CNT; ++k) M.red[i][rbase + k] = lsum[k];
    if (!group_sync()) return;
    const size_t pi = panel_index(a, x);
    if (gt < a.R) {
      const float l = (M.red[0][gt] + M.red[1][gt]) + (M.red[2][gt] + M.red[3][gt]);
      a.panel_ml[pi + gt] = make_float2(l > 0.f ? M.mref[gt] : -INFINITY, l);
    }
    if (!mbar_wait(&M.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort)) return;
    tc_fence_after();
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
#pragma unroll
      for (int c16 = 0; c16 < NM / 16; ++c16) {
        uint32_t r[16];
        tmem_load16(lane_base + kColO + 64 * h + 16 * c16, r);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int row = 16 * c16 + k;
          if (row < a.R) a.panel_o[(pi + row) * Fmt::D + h * 128 + gt] = __uint_as_float(r[k]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.o_free);
    if (!group_sync()) return;
    if (gt < kMaxRows) {
      M.mref[gt] = kNoMax;
      M.thr[gt] = -INFINITY;
    }
    if (!group_sync()) return;
  }
}

template <class Fmt, int NM, int TMA>
__global__ void __launch_bounds__(kThreads, 1) split_kernel(const __grid_constant__ SplitArgs a) {
  uint8_t* sm = smem_base();
  Misc& M = *reinterpret_cast<Misc*>(sm + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&M.kst_full[s], a.use_tma ? 1 : 32);
      mbar_init(&M.vst_full[s], a.use_tma ? 1 : 32);
      mbar_init(&M.kst_empty[s], 32);
      mbar_init(&M.vst_empty[s], 32);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&M.kbuf_full[s], 4);
      mbar_init(&M.kbuf_empty[s], 1);
      mbar_init(&M.s_full[s], 1);
      mbar_init(&M.s_empty[s], 4);
      mbar_init(&M.p_full[s], 4);
      mbar_init(&M.pv_done[s], 1);
    }
    mbar_init(&M.vbuf_full, 4);
    mbar_init(&M.q_full, 1);
    mbar_init(&M.q_empty, 1);
    mbar_init(&M.o_free, 4);
    mbar_init(&M.grp, 4);
    mbar_init(&M.fin, 1);
    M.ctl.abort = 0;
    M.ctl.limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimitCycles;
    M.rescale_tag = 0;
    for (int w = 0; w < 8; ++w) M.exceed_tag[w / 4][w % 4] = 0;
    mbar_fence_init();
  }
  if (tid < kMaxRows) {
    M.mref[tid] = kNoMax;
    M.thr[tid] = -INFINITY;
  }
  if (warp == 1) tmem_alloc(&M.tmem_base, 512);
  // zero the Q tile (rows >= R stay zero) and both P^T buffers (rows >= N stay zero)
  for (int o = tid * 16; o < 32768; o += kThreads * 16) *reinterpret_cast<uint4*>(sm + kOffQ + o) = make_uint4(0, 0, 0, 0);
  for (int o = tid * 16; o < 32768; o += kThreads * 16) *reinterpret_cast<uint4*>(sm + kOffP + o) = make_uint4(0, 0, 0, 0);
  sched_build(M.sched, a.ctx_lens, a.B, a.Hkv, a.max_ctx, a.status, a.bad);  // contains __syncthreads
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = M.tmem_base;

  if (warp == 0) {
    role_loader<TMA>(a, M, false, lane);
  } else if (warp == 2) {
    role_loader<TMA>(a, M, true, lane);
  } else if (warp == 3) {
    role_qload<Fmt>(a, M, lane);
  } else if (warp == 1) {
    if (lane == 0) {
      role_mma<Fmt, NM>(a, M, tb);
      // drain: every issued MMA must finish before TMEM is released
      mma_commit(&M.fin);
      const long long t0 = clock64();
      while (!mbar_try_wait(&M.fin, 0) && clock64() - t0 < M.ctl.limit) {
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    role_kdecode<Fmt>(a, M, warp - 4, lane, tb);
  } else if (warp < 12) {
    role_vdecode<Fmt>(a, M, warp - 8, lane);
  } else {
    role_softmax<Fmt, NM>(a, M, warp - 12, lane, tb);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
  if (tid == 0 && M.ctl.abort) atomicOr(a.status, 0x4u);
}

template <class Fmt, int NM, int TMA>
cudaError_t launch_one(const SplitArgs& a, int grid, cudaStream_t stream) {
  auto kern = split_kernel<Fmt, NM, TMA>;
  // the attribute is per device; setting it is idempotent, so a racing second
  // setter is harmless
  static std::atomic<uint64_t> set_on_devices{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(set_on_devices.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    set_on_devices.fetch_or(bit);
  }
  kern<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
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

int split_smem_bytes() { return kSmemBytes; }

cudaError_t launch_split(const SplitArgs& a, bool bf16, int grid, cudaStream_t stream) {
  if (bf16) return a.use_tma ? launch_mode<Bf16Fmt, 1>(a, grid, stream) : launch_mode<Bf16Fmt, 0>(a, grid, stream);
  return a.use_tma ? launch_mode<Fp8Fmt, 1>(a, grid, stream) : launch_mode<Fp8Fmt, 0>(a, grid, stream);
}

}  // namespace pa
