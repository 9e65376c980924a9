// Causal prefill attention, FP16 Q/K/V at head_dim 256, on sm_103a: tcgen05
// products with FP32 accumulation in tensor memory, TMA staging, and an
// online softmax whose reference max moves lazily.
//
// What it computes ("SM70 attention and quantized projection coverage across
// TP sizes", sections "Scope" and "Accumulation audit and rejected tuning":
// the Q8192 x KV262144 causal prefill with FP16 inputs and intermediates and
// FP32 accumulation for both QK and PV): for request b, query i < q_len and
// query head h (KV head h / G), query i sees keys 0 .. kv_len - q_len + i
// (the queries are the last q_len positions of the context), and
//   out = sum_j 2^(x_j - m) v_j / sum_j 2^(x_j - m),  x_j = (q . k_j) log2(e) / 16,
// which is the softmax of q . k_j / sqrt(256) in base 2.
//
// Work decomposition: one CTA per SM, persistent over work items.  An item
// is (request, query head, tile of 128 queries, key split of split_len keys);
// it writes FP32 partials (unnormalised O, reference max m, sum l) for its
// 128 rows, and a second kernel merges each row's splits in ascending order.
// The split length depends on kv_len alone, so a row's bits do not depend
// on the batch or head count.
//
// Roles (224 threads):
//   warps 0-3  softmax: thread = query row = TMEM lane; the item's Q rows
//              into TMEM; O rescale; epilogue
//   warp 4     TMA loader (one thread): K and V pieces of 16 KB into a
//              ring, in the order they are consumed
//   warp 5     TMEM allocation and the QK issuer (one thread)
//   warp 6     the PV issuer (one thread)
// TMEM (512 columns): the Q tile at columns 0-127 (FP16, two d per column),
// S at 128 (128 rows x 128 keys, FP32), O at 256 (128 rows x 256 d, FP32).
// Shared memory: P double buffer (2 x 32 KB, FP16), ring of 10 K/V pieces.
//   S(j)  = Q K(j)^T   A = Q (TMEM), B = K piece (shared, K-major), M 128,
//                      N 128, 16 steps of K 16 over d
//   O    += P(j) V(j)  A = P (shared, K-major), B = V piece (shared,
//                      MN-major), M 128, N 256, 8 steps of K 16 over keys
// The tensor core computes S(j+1) while the softmax works on S(j): S is free
// again once the softmax has read it into registers, and P has buffers of
// its own.  With Q in TMEM the QK products read only K from shared memory;
// the shared-memory traffic (TMA writes of K and V, P writes, operand reads)
// is what bounds this kernel.
#include <cuda_fp16.h>

#include <atomic>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kPfThreads = 224;
constexpr int kPfRows = 128;      // queries per tile (M)
constexpr int kPfKeys = 128;      // keys per tile
constexpr int kPfRing = 10;       // ring pieces
constexpr int kPfPiece = 16384;   // one K piece (128 keys x 64 d) or V piece (32 keys x 256 d)
constexpr int kPfPBytes = 32768;  // one P buffer: 2 atoms of 128 queries x 64 keys (FP16)
constexpr float kPfTau = 8.0f;    // the reference max moves only when a score exceeds it by 2^8
constexpr float kPfNoMax = -1e30f;  // reference max of a row that has seen no key (finite, so 2^(x - m) is never NaN)
constexpr uint32_t kPfColQ = 0;
constexpr uint32_t kPfColS = 128;
constexpr uint32_t kPfColO = 256;

struct PfBars {
  uint64_t full[kPfRing], empty[kPfRing];
  uint64_t q_full, s_full, s_free, p_full[2], pv_done[2], o_full, o_free, fin_qk, fin_pv;
  uint32_t tmem_base;
  WaitCtl ctl;
};

constexpr int kPfOffP = 0;
constexpr int kPfOffRing = kPfOffP + 2 * kPfPBytes;
constexpr int kPfOffBars = kPfOffRing + kPfRing * kPfPiece;
constexpr int kPfSmem = kPfOffBars + (int)sizeof(PfBars) + 1024;  // + slack for the 1024-byte alignment
static_assert(kPfSmem <= 232448, "prefill shared memory map exceeds the per-block limit");

__device__ __forceinline__ uint8_t* pf_smem() {
  extern __shared__ uint8_t pf_smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

struct PfItem {
  int b, h, qt, s, k0, k1, nt;
};

// Item it = ((s * B + b) * n_qt + qt) * Hq + h.  Its keys are [k0, k1): the
// split's keys up to the last key any row of the tile sees; nt tiles of 128.
__device__ __forceinline__ PfItem pf_item(const PrefillArgs& a, int it) {
  PfItem x;
  x.h = it % a.Hq;
  int t = it / a.Hq;
  x.qt = t % a.n_qt;
  t /= a.n_qt;
  x.b = t % a.B;
  x.s = t / a.B;
  x.k0 = x.s * a.split_len;
  const long long vis = (long long)a.kv_len - a.q_len + (long long)(x.qt + 1) * kPfRows;
  const int kend = vis <= 0 ? 0 : (vis < a.kv_len ? (int)vis : a.kv_len);
  x.k1 = min(x.k0 + a.split_len, kend);
  x.nt = x.k1 > x.k0 ? (x.k1 - x.k0 + kPfKeys - 1) / kPfKeys : 0;
  return x;
}

// Loader: per item the pieces with K two tiles ahead of V: K(0), K(1), then
// K(j), V(j-2) for j = 2 .. nt-1, then the last two V.  K(j) = 4 pieces (d
// atoms), V(j) = 4 pieces (32 keys each).  With K ahead, the ring never
// holds back QK(j+2) behind PV(j), which waits for the softmax.  Keys past
// kv_len arrive as zeros (outside the view).
__device__ void pf_loader(const PrefillArgs& a, PfBars& M, uint8_t* sm) {
  WaitCtl* ctl = &M.ctl;
  const uint32_t ring0 = smem_u32(sm + kPfOffRing);
  uint32_t f = 0;  // pieces issued
  int n = 0;       // items started
  for (int it = blockIdx.x; it < a.total_items; it += gridDim.x) {
    const PfItem x = pf_item(a, it);
    if (x.nt == 0) continue;
    ++n;
    const int g = x.h / a.G;
    bool ok = true;
    auto piece = [&](bool is_v, int j, int part) -> bool {
      const uint32_t slot = f % kPfRing, use = f / kPfRing;
      if (!mbar_wait(&M.empty[slot], (use & 1) ^ 1, ctl)) return false;
      const uint32_t dst = ring0 + slot * kPfPiece;
      const int kb = x.k0 + j * kPfKeys;
      if (is_v)
        tma_load_5d(dst, &a.v_map, 0, kb + 32 * part, 0, g, x.b, &M.full[slot]);
      else
        tma_load_4d(dst, &a.k_map, 64 * part, g, kb, x.b, &M.full[slot]);
      mbar_arrive_expect_tx(&M.full[slot], kPfPiece);
      ++f;
      return true;
    };
    for (int j = 0; ok && j < 2 && j < x.nt; ++j)
      for (int p = 0; ok && p < 4; ++p) ok = piece(false, j, p);
    for (int j = 2; ok && j < x.nt; ++j) {
      for (int p = 0; ok && p < 4; ++p) ok = piece(false, j, p);
      for (int p = 0; ok && p < 4; ++p) ok = piece(true, j - 2, p);
    }
    for (int j = x.nt > 2 ? x.nt - 2 : 0; ok && j < x.nt; ++j)
      for (int p = 0; ok && p < 4; ++p) ok = piece(true, j, p);
    if (!ok) break;
  }
  if (ctl->abort) {
    // let this thread's copies in flight land before the CTA exits
    if (f > 0) mbar_drain(&M.full[(f - 1) % kPfRing], ((f - 1) / kPfRing) & 1, ctl);
  }
}

// Fill index (within an item whose first piece is fill f0) of the first
// piece of K(j) and of V(j), in the loader's order K(0), K(1), [K(j),
// V(j-2)] for j >= 2, V(nt-2), V(nt-1): four pieces each.
__device__ __forceinline__ uint32_t pf_fill_k(uint32_t f0, int j) {
  return j == 0 ? f0 : (j == 1 ? f0 + 4u : f0 + 8u * j - 8u);
}
__device__ __forceinline__ uint32_t pf_fill_v(uint32_t f0, int j, int nt) {
  return j + 3 <= nt ? f0 + 12u + 8u * j : f0 + 8u * nt - 4u * (nt - j);
}

// QK issuer (one thread): S(j) = Q K(j)^T over 4 pieces (d atoms) of 4
// steps each, once the softmax has written the item's Q rows into TMEM and
// has read S(j-1) out of the S columns.  Each ring piece is released by a
// commit after the products that read it.  The two issuers run on separate threads so that
// their instruction streams overlap (one thread issues an MMA every 100 or
// so cycles, slower than the tensor core runs these shapes).
__device__ void pf_mma_qk(const PrefillArgs& a, PfBars& M, uint8_t* sm, uint32_t tb) {
  constexpr uint32_t id_qk = idesc_f16(128, 128, 0, 0, 0);
  WaitCtl* ctl = &M.ctl;
  const uint32_t ring0 = smem_u32(sm + kPfOffRing);
  uint32_t f0 = 0, jg = 0;  // first fill of the item, tiles of earlier items
  int n = 0;                // items started
  for (int it = blockIdx.x; it < a.total_items; it += gridDim.x) {
    const PfItem x = pf_item(a, it);
    if (x.nt == 0) continue;
    if (!mbar_wait(&M.q_full, n & 1, ctl)) return;
    tc_fence_after();
    for (int j = 0; j < x.nt; ++j) {
      const uint32_t jj = jg + j;
      if (jj >= 1 && !mbar_wait(&M.s_free, (jj - 1) & 1, ctl)) return;
      const uint32_t s_col = tb + kPfColS;
      const uint32_t fk = pf_fill_k(f0, j);
      for (int at = 0; at < 4; ++at) {
        const uint32_t idx = fk + at, slot = idx % kPfRing, use = idx / kPfRing;
        if (!mbar_wait(&M.full[slot], use & 1, ctl)) return;
        tc_fence_after();
        const uint64_t k_desc = sdesc_sw128(ring0 + slot * kPfPiece, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(s_col, tb + kPfColQ + (uint32_t)(4 * at + kk) * 8, sdesc_add(k_desc, kk * 32), id_qk,
                 (at | kk) != 0 ? 1u : 0u);
        mma_commit(&M.empty[slot]);
      }
      mma_commit(&M.s_full);
    }
    f0 += 8u * x.nt;
    jg += x.nt;
    ++n;
  }
}

// PV issuer (one thread): O += P(j) V(j) over 4 pieces (32 keys) of 2 steps
// each, P(j) from shared buffer j & 1 once the softmax has written it; an
// item's first product overwrites O once the previous item's epilogue has
// read it.
__device__ void pf_mma_pv(const PrefillArgs& a, PfBars& M, uint8_t* sm, uint32_t tb) {
  constexpr uint32_t id_pv = idesc_f16(128, 256, 0, 0, 1);
  WaitCtl* ctl = &M.ctl;
  const uint32_t ring0 = smem_u32(sm + kPfOffRing);
  const uint32_t p0 = smem_u32(sm + kPfOffP);
  uint32_t f0 = 0, jg = 0;
  int n = 0;
  for (int it = blockIdx.x; it < a.total_items; it += gridDim.x) {
    const PfItem x = pf_item(a, it);
    if (x.nt == 0) continue;
    for (int j = 0; j < x.nt; ++j) {
      const uint32_t jj = jg + j;
      if (!mbar_wait(&M.p_full[jj & 1], (jj >> 1) & 1, ctl)) return;
      if (j == 0 && !mbar_wait(&M.o_free, (n & 1) ^ 1, ctl)) return;
      tc_fence_after();
      const uint64_t p_desc = sdesc_sw128(p0 + (jj & 1) * kPfPBytes, 16, 1024);
      const uint32_t fv = pf_fill_v(f0, j, x.nt);
      for (int pc = 0; pc < 4; ++pc) {
        const uint32_t idx = fv + pc, slot = idx % kPfRing, use = idx / kPfRing;
        if (!mbar_wait(&M.full[slot], use & 1, ctl)) return;
        tc_fence_after();
        const uint64_t v_desc = sdesc_sw128(ring0 + slot * kPfPiece, 4096, 1024);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          // keys 32 pc + 16 kk .. +15: atom pc / 2, 32-byte step (2 pc + kk) % 4 within it
          const uint32_t p_off = (uint32_t)(pc >> 1) * 16384u + (uint32_t)((2 * pc + kk) & 3) * 32u;
          mma_ss(tb + kPfColO, sdesc_add(p_desc, p_off), sdesc_add(v_desc, kk * 2048), id_pv,
                 (j > 0 || pc > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&M.empty[slot]);
      }
      mma_commit(&M.pv_done[jj & 1]);
      if (j == x.nt - 1) mma_commit(&M.o_full);
    }
    f0 += 8u * x.nt;
    jg += x.nt;
    ++n;
  }
}

// Softmax, one query row per thread (row r = TMEM lane r).  Per tile: load
// the 128 scores and release the S buffer, mask keys the row does not see,
// take the tile max; the item's first tile sets the reference max m, a later
// tile moves it only when its max exceeds m by 2^kPfTau (then O, after
// PV(j-1), and l are scaled by 2^(m_old - m_new)); write P = 2^(x - m) in
// FP16 into shared P buffer j & 1 (once PV(j-2) has read it), K-major with
// the 128-byte swizzle (row r's 16-byte chunk c of atom a at a * 16384 +
// r * 128 + ((c ^ (r % 8)) * 16)), and add it to l.  After the item's last
// PV: the row's partial (O, m, l) to global memory.
// The TMEM loads and stores are warp-wide instructions, so every decision
// that leads to one is taken by the whole warp: a rescale runs for all 32
// rows when any of them needs it (the others with the factor 1, which leaves
// their bits unchanged), and a failed wait on any lane ends the whole warp.
__device__ void pf_softmax(const PrefillArgs& a, PfBars& M, int warp, int lane, uint32_t tb, uint8_t* sm) {
  WaitCtl* ctl = &M.ctl;
  const int r = warp * 32 + lane;
  const uint32_t lane_base = tb + ((uint32_t)(warp * 32) << 16);
  const float scale = 1.4426950408889634f / 16.0f;  // log2(e) / sqrt(256)
  uint32_t jg = 0;
  int n = 0;
  for (int it = blockIdx.x; it < a.total_items; it += gridDim.x) {
    const PfItem x = pf_item(a, it);
    if (x.nt == 0) continue;
    // keys t < vis_end are visible to this row within the item
    const long long lim = (long long)a.kv_len - a.q_len + (long long)x.qt * kPfRows + r + 1;
    const long long vis_end = lim < x.k1 ? lim : x.k1;
    float m_ref = kPfNoMax, l = 0.0f;
    // the item's Q row into TMEM columns 0-127 (query 128 qt + r of head h,
    // zeros past q_len); every QK of the previous item has completed (its
    // last S was read before this point)
    {
      const int qi = x.qt * kPfRows + r;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __half*>(a.q) +
                                                        (((size_t)x.b * a.q_len + qi) * a.Hq + x.h) * 256);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 v4 = qi < a.q_len ? __ldg(src + 4 * c + e) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * e] = v4.x, w[4 * e + 1] = v4.y, w[4 * e + 2] = v4.z, w[4 * e + 3] = v4.w;
        }
        PA_TMEM_ST_X16(lane_base + kPfColQ + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.q_full);
    }
    for (int j = 0; j < x.nt; ++j, ++jg) {
      if (!__all_sync(0xffffffffu, mbar_wait(&M.s_full, jg & 1, ctl))) return;
      tc_fence_after();
      const uint32_t s_addr = lane_base + kPfColS;
      uint32_t u[128];
#pragma unroll
      for (int c = 0; c < 8; ++c) PA_TMEM_LD_X16(s_addr + 16 * c, (u + 16 * c));
      tmem_wait_ld();
      reg_fence(u);
      // S(j) is in registers: QK(j+1) may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.s_free);
      const long long t0 = (long long)x.k0 + (long long)j * kPfKeys;
      const long long nv = vis_end - t0;
      const int nvis = nv <= 0 ? 0 : (nv >= kPfKeys ? kPfKeys : (int)nv);
      float v[128];
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
      if (nvis == kPfKeys) {
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          v[c] = __uint_as_float(u[c]) * scale;
          v[c + 1] = __uint_as_float(u[c + 1]) * scale;
          v[c + 2] = __uint_as_float(u[c + 2]) * scale;
          v[c + 3] = __uint_as_float(u[c + 3]) * scale;
          mx0 = fmaxf(mx0, v[c]), mx1 = fmaxf(mx1, v[c + 1]), mx2 = fmaxf(mx2, v[c + 2]), mx3 = fmaxf(mx3, v[c + 3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          v[c] = c < nvis ? __uint_as_float(u[c]) * scale : -INFINITY;
          v[c + 1] = c + 1 < nvis ? __uint_as_float(u[c + 1]) * scale : -INFINITY;
          v[c + 2] = c + 2 < nvis ? __uint_as_float(u[c + 2]) * scale : -INFINITY;
          v[c + 3] = c + 3 < nvis ? __uint_as_float(u[c + 3]) * scale : -INFINITY;
          mx0 = fmaxf(mx0, v[c]), mx1 = fmaxf(mx1, v[c + 1]), mx2 = fmaxf(mx2, v[c + 2]), mx3 = fmaxf(mx3, v[c + 3]);
        }
      }
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const bool up = j > 0 && mt > m_ref + kPfTau;
      if (j == 0) {
        m_ref = fmaxf(mt, kPfNoMax);
      } else if (__any_sync(0xffffffffu, up)) {
        const float alpha = up ? ex2_approx(m_ref - mt) : 1.0f;
        // O holds PV(0 .. j-1) once PV(j-1) has completed
        if (!__all_sync(0xffffffffu, mbar_wait(&M.pv_done[(jg - 1) & 1], ((jg - 1) >> 1) & 1, ctl))) return;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {
          uint32_t o[16];
          tmem_load16(lane_base + kPfColO + 16 * c, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          PA_TMEM_ST_X16(lane_base + kPfColO + 16 * c, o);
        }
        if (up) {
          l *= alpha;
          m_ref = mt;
        }
      }
      uint32_t pk[64];
      float l0 = 0.0f, l1 = 0.0f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2_approx(v[2 * c] - m_ref);
        const float p1 = ex2_approx(v[2 * c + 1] - m_ref);
        l0 += p0, l1 += p1;
        const __half2 h2 = __floats2half2_rn(p0, p1);
        pk[c] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      l += l0 + l1;
      // P buffer jg & 1 is free once PV(jg-2) has completed
      if (jg >= 2 && !__all_sync(0xffffffffu, mbar_wait(&M.pv_done[jg & 1], ((jg - 2) >> 1) & 1, ctl))) return;
      uint8_t* prow = sm + kPfOffP + (jg & 1) * kPfPBytes + r * 128;
#pragma unroll
      for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + a2 * 16384 + ((c ^ (r & 7)) << 4)) =
              make_uint4(pk[32 * a2 + 4 * c], pk[32 * a2 + 4 * c + 1], pk[32 * a2 + 4 * c + 2], pk[32 * a2 + 4 * c + 3]);
      tmem_wait_st();  // the O rescale's stores, if any
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.p_full[jg & 1]);
    }
    // epilogue: the row's partial, then O is free for the next item
    if (!__all_sync(0xffffffffu, mbar_wait(&M.o_full, n & 1, ctl))) return;
    tc_fence_after();
    const size_t pidx = (((size_t)x.b * a.Hq + x.h) * a.n_qt + x.qt) * a.num_splits + x.s;
    float4* po = reinterpret_cast<float4*>(a.part_o + (pidx * kPfRows + r) * 256);
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {
      uint32_t o[16];
      tmem_load16(lane_base + kPfColO + 16 * c, o);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        po[4 * c + e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                    __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
    }
    a.part_ml[pidx * kPfRows + r] = make_float2(m_ref, l);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.o_free);
    ++n;
  }
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  uint8_t* sm = pf_smem();
  PfBars& M = *reinterpret_cast<PfBars*>(sm + kPfOffBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kPfRing; ++s) {
      mbar_init(&M.full[s], 1);
      mbar_init(&M.empty[s], 1);
    }
    mbar_init(&M.q_full, 4);  // one arrival per softmax warp
    mbar_init(&M.s_full, 1);
    mbar_init(&M.s_free, 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&M.p_full[s], 4);  // one arrival per softmax warp
      mbar_init(&M.pv_done[s], 1);
    }
    mbar_init(&M.o_full, 1);
    mbar_init(&M.o_free, 4);
    mbar_init(&M.fin_qk, 1);
    mbar_init(&M.fin_pv, 1);
    M.ctl.abort = 0;
    M.ctl.limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimitCycles;
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(&M.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = M.tmem_base;

  if (warp < 4) {
    pf_softmax(a, M, warp, lane, tb, sm);
  } else if (warp == 4) {
    if (lane == 0) pf_loader(a, M, sm);
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      pf_mma_qk(a, M, sm, tb);
      // every product this thread issued completes before TMEM is released
      mma_commit(&M.fin_qk);
      mbar_drain(&M.fin_qk, 0, &M.ctl);
    }
    __syncwarp();
  } else {
    if (lane == 0) {
      pf_mma_pv(a, M, sm, tb);
      mma_commit(&M.fin_pv);
      mbar_drain(&M.fin_pv, 0, &M.ctl);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
  if (tid == 0 && M.ctl.abort) atomicOr(a.status, 0x4u);
}

// One warp per output row (request b, query i, head h); lane l holds d
// 8l .. 8l+7.  Splits are merged in ascending order with weights
// 2^(m_s - max m): O = sum w_s O_s / sum w_s l_s, LSE = (max m + log2 L) ln 2.
// A row that sees no key is written as zeros with LSE -inf.
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillMergeArgs m) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + warp;
  if (row >= (long long)m.B * m.q_len * m.Hq) return;
  const int h = (int)(row % m.Hq);
  const long long t = row / m.Hq;
  const int i = (int)(t % m.q_len), b = (int)(t / m.q_len);
  const int qt = i / kPfRows, r = i % kPfRows;
  const long long vis = (long long)m.kv_len - m.q_len + (long long)(qt + 1) * kPfRows;
  const int kend = vis <= 0 ? 0 : (vis < m.kv_len ? (int)vis : m.kv_len);
  const int ns = (kend + m.split_len - 1) / m.split_len;
  const size_t base = (((size_t)b * m.Hq + h) * m.n_qt + qt) * m.num_splits;
  float mmax = kPfNoMax;
  for (int s = 0; s < ns; ++s) mmax = fmaxf(mmax, m.part_ml[(base + s) * kPfRows + r].x);
  float L = 0.0f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < ns; ++s) {
    const float2 ml = m.part_ml[(base + s) * kPfRows + r];
    const float w = exp2f(ml.x - mmax);
    L = fmaf(w, ml.y, L);
    const float4* po = reinterpret_cast<const float4*>(m.part_o + ((base + s) * kPfRows + r) * 256 + 8 * lane);
    const float4 a0 = __ldcs(po), a1 = __ldcs(po + 1);
    acc[0] = fmaf(w, a0.x, acc[0]), acc[1] = fmaf(w, a0.y, acc[1]);
    acc[2] = fmaf(w, a0.z, acc[2]), acc[3] = fmaf(w, a0.w, acc[3]);
    acc[4] = fmaf(w, a1.x, acc[4]), acc[5] = fmaf(w, a1.y, acc[5]);
    acc[6] = fmaf(w, a1.z, acc[6]), acc[7] = fmaf(w, a1.w, acc[7]);
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2 h2 = __floats2half2_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    o[e] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(m.out) + row * 256 + 8 * lane);
  *dst = make_uint4(o[0], o[1], o[2], o[3]);
  if (m.lse != nullptr && lane == 0)
    m.lse[row] = L > 0.0f ? (mmax + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

int prefill_smem_bytes() { return kPfSmem; }

cudaError_t launch_prefill(const PrefillArgs& a, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> set_on_devices{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(set_on_devices.load() & bit)) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return e;
    set_on_devices.fetch_or(bit);
  }
  prefill_kernel<<<grid, kPfThreads, kPfSmem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_merge(const PrefillMergeArgs& m, cudaStream_t stream) {
  const long long rows = (long long)m.B * m.q_len * m.Hq;
  if (rows <= 0) return cudaSuccess;
  prefill_merge_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(m);
  return cudaGetLastError();
}

}  // namespace pa
