// C ABI of libpa (declared in include/pa.h): host-side validation, workspace
// layout, launches and the timing / bookkeeping helpers.  No device memory is
// allocated here; every buffer belongs to the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "pa.h"
#include "plan.cuh"

namespace {

using namespace pa;

constexpr int kMaxDevices = 64;

// Test hook state (pa_debug_stall_next): the next decode call runs with this
// wait bound and withholds its Q-ready signal.
std::atomic<long long> g_stall_next{0};

int sm_count(int dev) {
  static std::mutex mu;
  static int cache[kMaxDevices] = {0};
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Geometry checks shared by every decode call.  *R receives G * q_len.
int check_geometry(const pa_params* p, int head_dim, int* R) {
  if (p == nullptr) return PA_ERR_NULL;
  if (p->head_dim != head_dim) return PA_ERR_UNSUPPORTED;
  if (p->batch < 1 || p->batch > kMaxBatch) return PA_ERR_SHAPE;
  if (p->num_kv_heads < 1 || p->num_q_heads < 1 || p->num_q_heads % p->num_kv_heads != 0) return PA_ERR_SHAPE;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G > kMaxGroup) return PA_ERR_UNSUPPORTED;
  if (p->q_len < 1 || p->q_len > kMaxQLen) return PA_ERR_SHAPE;
  if (G * p->q_len > kMaxRows) return PA_ERR_UNSUPPORTED;
  if (p->page_size <= 0 || p->page_size % kPageMultiple != 0) return PA_ERR_SHAPE;
  if (p->max_ctx_len < 0 || p->max_ctx_len > kMaxCtx) return PA_ERR_SHAPE;
  if (p->num_pages < 1 || p->max_pages_per_req < 1) return PA_ERR_SHAPE;
  if ((long long)p->max_pages_per_req * p->page_size < (long long)p->max_ctx_len) return PA_ERR_SHAPE;
  const long long st[6] = {p->k_page_stride, p->k_token_stride, p->k_head_stride,
                           p->v_page_stride, p->v_token_stride, p->v_head_stride};
  for (long long s : st) {
    if (s < 0) return PA_ERR_SHAPE;
    if (s % 8 != 0) return PA_ERR_ALIGN;
  }
  *R = G * p->q_len;
  return PA_OK;
}

size_t workspace_bytes(const pa_params* p, int head_dim) {
  int R = 0;
  if (check_geometry(p, head_dim, &R) != PA_OK) return 0;
  return ws_layout(p->batch, p->num_kv_heads, max_splits_for(p->max_ctx_len), R, head_dim).total;
}

bool strides16(const pa_params* p) {
  return p->k_page_stride % 16 == 0 && p->k_token_stride % 16 == 0 && p->k_head_stride % 16 == 0 &&
         p->v_page_stride % 16 == 0 && p->v_token_stride % 16 == 0 && p->v_head_stride % 16 == 0;
}

// K/V load path from alignment alone (the tensor-map encoder may still refuse)
KvLoad kv_load_for(const pa_params* p, const void* k, const void* v) {
  if (!strides16(p)) return kKvLoadCopy;
  if (aligned(k, 16) && aligned(v, 16)) return kKvLoadTma;
  const uintptr_t km = reinterpret_cast<uintptr_t>(k) % 16, vm = reinterpret_cast<uintptr_t>(v) % 16;
  return km == 8 && vm == 8 ? kKvLoadWindow : kKvLoadCopy;
}

// ---- TMA tensor maps ----------------------------------------------------------
// The CUDA driver API's tensor-map encoder, fetched through the runtime so the library
// does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D byte view of K or V: (row byte 0..row_bytes-1, KV head, slot, page),
// boxes of 128 bytes x 1 head x `slots` slots, 128-byte swizzle.  A box taller
// than a page is clipped to the page (the loader never uses a box taller than
// the piece of a page it copies).
bool encode_kv_map(CUtensorMap* m, const void* base, const pa_params* p, bool v, unsigned slots, int row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const long long hs = v ? p->v_head_stride : p->k_head_stride;
  const long long ts = v ? p->v_token_stride : p->k_token_stride;
  const long long ps = v ? p->v_page_stride : p->k_page_stride;
  cuuint64_t dims[4] = {(cuuint64_t)row_bytes, (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->page_size,
                        (cuuint64_t)p->num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)(p->num_kv_heads == 1 ? row_bytes : hs), (cuuint64_t)ts, (cuuint64_t)ps};
  cuuint32_t box[4] = {128, 1, slots < (unsigned)p->page_size ? slots : (cuuint32_t)p->page_size, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (cuuint64_t s : strides)
    if (s == 0 || s % 16 != 0 || s >= (1ull << 40)) return false;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D byte view of K or V: (row byte 0..127, KV head, slot, 128-byte part of
// the key row, page), one box of 128 bytes x 1 head x 128 slots x 2 parts,
// 128-byte swizzle.  The box lands as part 0 of its 128 slots, then part 1:
// a whole staging tile of the split kernel in one copy.  Used only for tiles
// inside one page (page_size >= 128).
bool encode_kv_tile_map(CUtensorMap* m, const void* base, const pa_params* p, bool v, int row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const long long hs = v ? p->v_head_stride : p->k_head_stride;
  const long long ts = v ? p->v_token_stride : p->k_token_stride;
  const long long ps = v ? p->v_page_stride : p->k_page_stride;
  cuuint64_t dims[5] = {128, (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->page_size, (cuuint64_t)(row_bytes / 128),
                        (cuuint64_t)p->num_pages};
  cuuint64_t strides[4] = {(cuuint64_t)(p->num_kv_heads == 1 ? row_bytes : hs), (cuuint64_t)ts, 128, (cuuint64_t)ps};
  cuuint32_t box[5] = {128, 1, (cuuint32_t)(p->page_size < 128 ? p->page_size : 128), 2, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  for (cuuint64_t s : strides)
    if (s == 0 || s % 16 != 0 || s >= (1ull << 40)) return false;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Window view of K or V whose base lies 8 bytes past a 16-byte boundary (all
// strides multiples of 16): 4-D view of 16-bit elements (row element, KV
// head, slot, page) that starts 8 bytes before the base, so row element e
// holds row bytes 2e - 8, 2e - 7, and a row spans row_bytes/2 + 4 elements.
// Boxes of 136 elements (272 bytes) x 1 head x `slots` slots, no swizzle: a
// box at element 128h lands the 8 bytes before row byte 256h, the 256 row
// bytes from there and 8 bytes past them, each key's 272 bytes one after the
// other.  Every byte read lies in a 16-byte granule that holds bytes of the
// row itself (the row starts at 8 mod 16 and ends at 8 mod 16), so the copy
// never touches memory outside the caller's rows' granules; elements past the
// view (the last 8 bytes of the last fill) are filled with zeros, not read.
bool encode_kv_window_map(CUtensorMap* m, const void* base, const pa_params* p, bool v, unsigned slots,
                          int row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const long long hs = v ? p->v_head_stride : p->k_head_stride;
  const long long ts = v ? p->v_token_stride : p->k_token_stride;
  const long long ps = v ? p->v_page_stride : p->k_page_stride;
  cuuint64_t dims[4] = {(cuuint64_t)(row_bytes / 2 + 4), (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->page_size,
                        (cuuint64_t)p->num_pages};
  // with one KV head the head stride is never applied; any multiple of 16 serves
  cuuint64_t strides[3] = {(cuuint64_t)(p->num_kv_heads == 1 ? row_bytes + 16 : hs), (cuuint64_t)ts, (cuuint64_t)ps};
  cuuint32_t box[4] = {136, 1, slots < (unsigned)p->page_size ? slots : (cuuint32_t)p->page_size, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (cuuint64_t s : strides)
    if (s == 0 || s % 16 != 0 || s >= (1ull << 40)) return false;
  void* start = const_cast<uint8_t*>(static_cast<const uint8_t*>(base) - 8);
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, start, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D element view of Q [B][q_len][Hq][D] (16-bit elements): (d, query head,
// verify query, request), boxes of 64 elements x G heads x q_len queries,
// 128-byte swizzle.  One box is one 64-column atom of an item's packed Q tile,
// rows in (verify query, head) order.
bool encode_q_map(CUtensorMap* m, const void* q, const pa_params* p, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const int G = p->num_q_heads / p->num_kv_heads;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p->num_q_heads, (cuuint64_t)p->q_len, (cuuint64_t)p->batch};
  const cuuint64_t row = (cuuint64_t)D * 2;
  cuuint64_t strides[3] = {row, row * p->num_q_heads, row * p->num_q_heads * p->q_len};
  cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)p->q_len, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- kernel timing ----------------------------------------------------------
struct Timing {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool[2];  // event pairs per kernel kind: [2*i], [2*i+1]
  size_t used[2] = {0, 0};
};
Timing& timing() {
  static Timing t;
  return t;
}
constexpr size_t kMaxTimed = 4096;

// Returns the two events to record around one launch of kernel `kind`, or
// {nullptr, nullptr} when timing is off or full.
void timing_slot(int kind, cudaEvent_t* a, cudaEvent_t* b) {
  *a = *b = nullptr;
  Timing& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  if (!T.on || T.used[kind] >= kMaxTimed) return;
  auto& pool = T.pool[kind];
  if (pool.size() < 2 * (T.used[kind] + 1)) {
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return;
    if (cudaEventCreate(&e1) != cudaSuccess) {
      cudaEventDestroy(e0);
      return;
    }
    pool.push_back(e0);
    pool.push_back(e1);
  }
  *a = pool[2 * T.used[kind]];
  *b = pool[2 * T.used[kind] + 1];
  T.used[kind]++;
}

// Fills the K/V tensor maps of the load path the alignment allows and returns
// that path, or kKvLoadCopy when the driver refuses an encoding.
KvLoad encode_kv_maps(SplitArgs* a, const pa_params* p, const void* k, const void* v, int row_bytes) {
  const KvLoad want = kv_load_for(p, k, v);
  bool ok = want != kKvLoadCopy;
  for (int m = 0; m < 4 && ok; ++m) {
    const unsigned slots = 128u >> m;
    ok = want == kKvLoadTma ? encode_kv_map(&a->k_maps[m], k, p, false, slots, row_bytes) &&
                                  encode_kv_map(&a->v_maps[m], v, p, true, slots, row_bytes)
                            : encode_kv_window_map(&a->k_maps[m], k, p, false, slots, row_bytes) &&
                                  encode_kv_window_map(&a->v_maps[m], v, p, true, slots, row_bytes);
  }
  if (ok && want == kKvLoadTma)
    ok = encode_kv_tile_map(&a->k_map_tile, k, p, false, row_bytes) &&
         encode_kv_tile_map(&a->v_map_tile, v, p, true, row_bytes);
  return ok ? want : kKvLoadCopy;
}

int decode_common(KvFormat fmt, const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale, const float* v_scale,
                  void* out, float* lse, void* workspace, size_t workspace_bytes_given, void* stream_ptr,
                  bool clear_status = false) {
  const bool scaled = fmt == kKvE4m3 || fmt == kKvE5m2;  // 8-bit K/V with FP32 per-tensor scales
  const int D = fmt == kKvBf16 ? 128 : 256;
  const int row_bytes = D * (scaled ? 1 : 2);
  int R = 0;
  int st = check_geometry(p, D, &R);
  if (st != PA_OK) return st;
  if (!q || !k_pages || !v_pages || !block_table || !ctx_lens || !out) return PA_ERR_NULL;
  if (scaled && (!k_scale || !v_scale)) return PA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 16))) return PA_ERR_ALIGN;
  if (!aligned(k_pages, 8) || !aligned(v_pages, 8) || !aligned(block_table, 4) || !aligned(ctx_lens, 4))
    return PA_ERR_ALIGN;
  if (scaled && (!aligned(k_scale, 4) || !aligned(v_scale, 4))) return PA_ERR_ALIGN;
  const int s_max = max_splits_for(p->max_ctx_len);
  const WsLayout L = ws_layout(p->batch, p->num_kv_heads, s_max, R, D);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes_given < L.total) return PA_ERR_WORKSPACE;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  const int nsm = sm_count(dev);
  if (nsm <= 0) return PA_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* bad = reinterpret_cast<uint32_t*>(ws + kWsBadOff);
  // the per-request flags, split arrival counters and task counters are zero
  // between calls (the workspace is zero at first use; the last CTA of every
  // call resets them), so a call is one launch
  if (clear_status && cudaMemsetAsync(status, 0, sizeof(uint32_t), stream) != cudaSuccess) return PA_ERR_CUDA;

  SplitArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = static_cast<const uint8_t*>(k_pages);
  a.v = static_cast<const uint8_t*>(v_pages);
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.panel_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  a.panel_o = reinterpret_cast<float*>(ws + L.o_off);
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.bad = bad;
  a.arrive = reinterpret_cast<uint32_t*>(ws + kWsArriveOff);
  a.queue = reinterpret_cast<uint32_t*>(ws + kWsQueueOff);
  a.done = reinterpret_cast<uint32_t*>(ws + kWsDoneOff);
  a.k_ps = p->k_page_stride, a.k_ts = p->k_token_stride, a.k_hs = p->k_head_stride;
  a.v_ps = p->v_page_stride, a.v_ts = p->v_token_stride, a.v_hs = p->v_head_stride;
  a.B = p->batch, a.Hkv = p->num_kv_heads, a.Hq = p->num_q_heads, a.G = p->num_q_heads / p->num_kv_heads;
  a.q_len = p->q_len, a.R = R, a.page_size = p->page_size, a.mpr = p->max_pages_per_req;
  a.num_pages = p->num_pages, a.max_ctx = p->max_ctx_len, a.s_max = s_max;
  // TMA boxes for 16-byte aligned K/V, TMA windows for bases 8 bytes past a
  // 16-byte boundary, cp.async for the rest (or where an encoding is refused)
  a.kv_load = encode_kv_maps(&a, p, k_pages, v_pages, row_bytes);
  // the packed Q tile by TMA together with K and V; with K/V by cp.async the
  // kernel runs its per-lane copy paths for all three
  a.q_tma = a.kv_load != kKvLoadCopy && encode_q_map(&a.q_map, q, p, D) ? 1 : 0;
  const long long stall = g_stall_next.exchange(0);
  a.wait_limit = stall > 0 ? stall : 0;
  a.withhold_q = stall > 0 ? 1 : 0;

  // one CTA per SM at most; at least as many as split items, and enough that
  // the merge phase's five workers per CTA take about one task (128 output
  // elements) each
  const long long max_items = (long long)p->batch * p->num_kv_heads * (s_max > 0 ? s_max : 1);
  const long long merge_ctas = ((long long)p->batch * p->num_kv_heads * R * (D / 128) + 4) / 5;
  const long long want = max_items > merge_ctas ? max_items : merge_ctas;
  const int grid = (int)(want < nsm ? want : nsm);
  cudaEvent_t e0, e1;
  timing_slot(0, &e0, &e1);
  if (e0) cudaEventRecord(e0, stream);
  if (launch_split(a, fmt, grid, stream) != cudaSuccess) return PA_ERR_CUDA;
  if (e1) cudaEventRecord(e1, stream);
  return PA_OK;
}

// ---- causal prefill -------------------------------------------------------------
constexpr int kPfMaxBatch = 64;
constexpr int kPfMaxQLen = 65536;
constexpr int kPfMaxKv = 1 << 22;
constexpr int kPfMaxHeads = 256;
constexpr int kPfTile = 128;

// split_len depends on kv_len alone: 32768 above 32768 keys, else kv_len / 8
// rounded up to whole 128-key tiles, at least 1024
void prefill_plan(int kv_len, int* num_splits, int* split_len) {
  int len = 32768;
  if (kv_len <= 32768) {
    len = ((kv_len + 7) / 8 + kPfTile - 1) / kPfTile * kPfTile;
    if (len < 1024) len = 1024;
  }
  *split_len = len;
  *num_splits = (kv_len + len - 1) / len;
}

struct PfLayout {
  size_t ml_off, o_off, total;
  long long tiles;  // (request, head, query tile, split) partial tiles
};

int check_prefill(const pa_prefill_params* p) {
  if (p == nullptr) return PA_ERR_NULL;
  if (p->head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (p->batch < 1 || p->batch > kPfMaxBatch || p->q_len < 1 || p->q_len > kPfMaxQLen || p->kv_len < 1 ||
      p->kv_len > kPfMaxKv)
    return PA_ERR_SHAPE;
  if (p->num_kv_heads < 1 || p->num_q_heads < 1 || p->num_q_heads > kPfMaxHeads ||
      p->num_q_heads % p->num_kv_heads != 0)
    return PA_ERR_SHAPE;
  const long long st[6] = {p->k_batch_stride, p->k_token_stride, p->k_head_stride,
                           p->v_batch_stride, p->v_token_stride, p->v_head_stride};
  const bool unit[6] = {p->batch == 1, false, p->num_kv_heads == 1, p->batch == 1, false, p->num_kv_heads == 1};
  for (int i = 0; i < 6; ++i) {
    if (unit[i]) continue;
    if (st[i] <= 0) return PA_ERR_SHAPE;
    if (st[i] % 8 != 0) return PA_ERR_ALIGN;
  }
  return PA_OK;
}

PfLayout prefill_layout(const pa_prefill_params* p) {
  int ns = 0, len = 0;
  prefill_plan(p->kv_len, &ns, &len);
  const long long n_qt = (p->q_len + kPfTile - 1) / kPfTile;
  PfLayout L;
  L.tiles = (long long)p->batch * p->num_q_heads * n_qt * ns;
  const size_t rows = (size_t)L.tiles * kPfTile;
  L.ml_off = 256;
  L.o_off = L.ml_off + (rows * sizeof(float2) + 255) / 256 * 256;
  L.total = L.o_off + rows * 256 * sizeof(float);
  return L;
}

// byte stride of a dimension; one of extent 1 is never applied, so any
// multiple of 16 serves
cuuint64_t pf_stride(long long elems, bool unit) { return unit ? 1024 : (cuuint64_t)elems * 2; }

bool encode_prefill_maps(PrefillArgs* a, const pa_prefill_params* p, const void* k, const void* v) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const auto il = CU_TENSOR_MAP_INTERLEAVE_NONE;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  const auto oob = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE;
  const bool b1 = p->batch == 1, h1 = p->num_kv_heads == 1;
  // K: (d, KV head, key, request)
  {
    cuuint64_t dims[4] = {256, (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->kv_len, (cuuint64_t)p->batch};
    cuuint64_t strides[3] = {pf_stride(p->k_head_stride, h1), pf_stride(p->k_token_stride, false),
                             pf_stride(p->k_batch_stride, b1)};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&a->k_map, f16, 4, const_cast<void*>(k), dims, strides, box, estr, il, sw, l2, oob) != CUDA_SUCCESS)
      return false;
  }
  // V: (d within atom, key, atom, KV head, request)
  {
    cuuint64_t dims[5] = {64, (cuuint64_t)p->kv_len, 4, (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->batch};
    cuuint64_t strides[4] = {pf_stride(p->v_token_stride, false), 128, pf_stride(p->v_head_stride, h1),
                             pf_stride(p->v_batch_stride, b1)};
    cuuint32_t box[5] = {64, 32, 4, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (enc(&a->v_map, f16, 5, const_cast<void*>(v), dims, strides, box, estr, il, sw, l2, oob) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

int prefill_f16(const pa_prefill_params* p, const void* q, const void* k, const void* v, void* out, float* lse,
                void* workspace, size_t workspace_bytes, void* stream_ptr) {
  int st = check_prefill(p);
  if (st != PA_OK) return st;
  if (!q || !k || !v || !out) return PA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
    return PA_ERR_ALIGN;
  const PfLayout L = prefill_layout(p);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  const int nsm = sm_count(dev);
  if (nsm <= 0) return PA_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_prefill_maps(&a, p, k, v)) return PA_ERR_CUDA;
  a.q = q;
  a.part_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  a.part_o = reinterpret_cast<float*>(ws + L.o_off);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.B = p->batch, a.q_len = p->q_len, a.kv_len = p->kv_len, a.Hq = p->num_q_heads, a.Hkv = p->num_kv_heads;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.n_qt = (p->q_len + kPfTile - 1) / kPfTile;
  prefill_plan(p->kv_len, &a.num_splits, &a.split_len);
  if (L.tiles > 0x7fffffffll) return PA_ERR_SHAPE;
  a.total_items = (int)L.tiles;
  a.wait_limit = 0;
  const int grid = a.total_items < nsm ? a.total_items : nsm;

  cudaEvent_t e0, e1;
  timing_slot(1, &e0, &e1);
  if (e0) cudaEventRecord(e0, stream);
  if (launch_prefill(a, grid, stream) != cudaSuccess) return PA_ERR_CUDA;
  if (e1) cudaEventRecord(e1, stream);
  PrefillMergeArgs m;
  m.part_o = a.part_o, m.part_ml = a.part_ml, m.out = out, m.lse = lse;
  m.B = a.B, m.q_len = a.q_len, m.kv_len = a.kv_len, m.Hq = a.Hq, m.n_qt = a.n_qt, m.split_len = a.split_len;
  m.num_splits = a.num_splits;
  if (launch_prefill_merge(m, stream) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

// ---- allocation-free variant ------------------------------------------------
// Scratch for pa_decode_fp8_noalloc: a module-scope device array that every
// device loading this library holds until the process exits.  Host code must
// not use its name as an address; the device address comes from
// cudaGetSymbolAddress with the calling device current.  It is looked up on
// every call rather than cached: the address belongs to the current context,
// and a cached value would outlive a cudaDeviceReset or a switch to another
// context on the same device.  Once the array's module is loaded the lookup
// is a table search in the runtime and allocates nothing.
constexpr size_t kNoallocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_get_capabilities(pa_caps* out) {
  if (out == nullptr) return PA_ERR_NULL;
  std::memset(out, 0, sizeof(*out));
  out->abi_version = PA_ABI_VERSION;
  out->max_batch = kMaxBatch;
  out->max_q_len = kMaxQLen;
  out->max_group = kMaxGroup;
  out->page_multiple = kPageMultiple;
  out->max_ctx = kMaxCtx;
  out->accum_bits = 32;
  out->fp8_head_dim = 256;
  out->bf16_head_dim = 128;
  out->max_splits = kMaxSplits;
  return PA_OK;
}

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_SHAPE: return "shape, length, page size or stride out of range";
    case PA_ERR_UNSUPPORTED: return "unsupported head_dim or GQA geometry";
    case PA_ERR_ALIGN: return "pointer or stride not aligned as required";
    case PA_ERR_WORKSPACE: return "workspace NULL, misaligned or too small";
    case PA_ERR_CUDA: return "CUDA runtime or launch failure";
    default: return "unknown status";
  }
}

int pa_split_plan(int32_t ctx_len, int32_t num_kv_heads, int32_t* num_splits, int32_t* chunk) {
  if (!num_splits || !chunk) return PA_ERR_NULL;
  if (ctx_len < 0 || num_kv_heads < 1) return PA_ERR_SHAPE;
  int s, c;
  split_plan(ctx_len, num_kv_heads, s, c);
  *num_splits = s;
  *chunk = c;
  return PA_OK;
}

size_t pa_decode_fp8_workspace_bytes(const pa_params* p) { return workspace_bytes(p, 256); }
size_t pa_decode_bf16_d128_workspace_bytes(const pa_params* p) { return workspace_bytes(p, 128); }

int pa_decode_fp8(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale, const float* v_scale,
                  void* out, void* workspace, size_t workspace_bytes_given, void* stream) {
  return decode_common(kKvE4m3, p, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out, nullptr,
                       workspace, workspace_bytes_given, stream);
}

int pa_decode_e5m2(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale, const float* v_scale,
                   void* out, void* workspace, size_t workspace_bytes_given, void* stream) {
  return decode_common(kKvE5m2, p, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out, nullptr,
                       workspace, workspace_bytes_given, stream);
}

int pa_decode_fp8_noalloc(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                          const float* v_scale, void* out, void* stream) {
  int R = 0;
  const int st = check_geometry(p, 256, &R);
  if (st != PA_OK) return st;
  if (workspace_bytes(p, 256) > kNoallocScratchBytes) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int sst = noalloc_scratch(&scratch);
  if (sst != PA_OK) return sst;
  return decode_common(kKvE4m3, p, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out, nullptr,
                       scratch, kNoallocScratchBytes, stream, /*clear_status=*/true);
}

int pa_decode_f16(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* ctx_lens, void* out, void* workspace,
                  size_t workspace_bytes_given, void* stream) {
  return decode_common(kKvF16, p, q, k_pages, v_pages, block_table, ctx_lens, nullptr, nullptr, out, nullptr,
                       workspace, workspace_bytes_given, stream);
}

int pa_decode_bf16_d256(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse, void* workspace,
                        size_t workspace_bytes_given, void* stream) {
  return decode_common(kKvBf16D256, p, q, k_pages, v_pages, block_table, ctx_lens, nullptr, nullptr, out, lse,
                       workspace, workspace_bytes_given, stream);
}

int pa_decode_bf16_d128(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse, void* workspace,
                        size_t workspace_bytes_given, void* stream) {
  return decode_common(kKvBf16, p, q, k_pages, v_pages, block_table, ctx_lens, nullptr, nullptr, out, lse, workspace,
                       workspace_bytes_given, stream);
}

int pa_prefill_plan(int32_t kv_len, int32_t* num_splits, int32_t* split_len) {
  if (!num_splits || !split_len) return PA_ERR_NULL;
  if (kv_len < 1) return PA_ERR_SHAPE;
  int ns = 0, len = 0;
  prefill_plan(kv_len, &ns, &len);
  *num_splits = ns;
  *split_len = len;
  return PA_OK;
}

size_t pa_prefill_f16_workspace_bytes(const pa_prefill_params* p) {
  if (check_prefill(p) != PA_OK) return 0;
  return prefill_layout(p).total;
}

int pa_prefill_f16(const pa_prefill_params* p, const void* q, const void* k, const void* v, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_f16(p, q, k, v, out, lse, workspace, workspace_bytes, stream);
}

int pa_read_status(const void* workspace, uint32_t* flags, void* stream) {
  if (!workspace || !flags) return PA_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

int pa_clear_status(void* workspace, void* stream) {
  if (!workspace) return PA_ERR_NULL;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_debug_worklist(const pa_params* p, const int32_t* ctx_lens, int32_t* items, int32_t max_items,
                      int32_t* count, void* stream) {
  if (!p || !ctx_lens || !items || !count) return PA_ERR_NULL;
  if (p->batch < 1 || p->batch > kMaxBatch || p->num_kv_heads < 1) return PA_ERR_SHAPE;
  if (p->max_ctx_len < 0 || p->max_ctx_len > kMaxCtx) return PA_ERR_SHAPE;
  const long long need = (long long)p->batch * p->num_kv_heads * max_splits_for(p->max_ctx_len);
  if (max_items < need) return PA_ERR_SHAPE;
  // invalid lengths are planned as 0 here too; the decode calls report them
  if (launch_debug_worklist(ctx_lens, p->batch, p->num_kv_heads, p->max_ctx_len, items, max_items, count,
                            nullptr, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_debug_gather_fp8(const pa_params* p, const void* k_pages, const void* v_pages, const int32_t* block_table,
                        const int32_t* ctx_lens, int32_t which, void* dst, void* stream) {
  int R = 0;
  int st = check_geometry(p, 256, &R);
  if (st != PA_OK) return st;
  if (!k_pages || !v_pages || !block_table || !ctx_lens || !dst) return PA_ERR_NULL;
  if (which != 0 && which != 1) return PA_ERR_SHAPE;
  const uint8_t* base = static_cast<const uint8_t*>(which == 0 ? k_pages : v_pages);
  const long long ps = which == 0 ? p->k_page_stride : p->v_page_stride;
  const long long ts = which == 0 ? p->k_token_stride : p->v_token_stride;
  const long long hs = which == 0 ? p->k_head_stride : p->v_head_stride;
  if (launch_debug_gather(base, ps, ts, hs, block_table, ctx_lens, p->batch, p->num_kv_heads, p->page_size,
                          p->max_pages_per_req, p->num_pages, p->max_ctx_len, 256, static_cast<uint8_t*>(dst),
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_debug_kv_load_path(const pa_params* p, int32_t head_dim, int32_t elem_bytes, const void* k_pages,
                          const void* v_pages, int32_t* path) {
  if (!p || !k_pages || !v_pages || !path) return PA_ERR_NULL;
  if ((head_dim != 128 && head_dim != 256) || (elem_bytes != 1 && elem_bytes != 2)) return PA_ERR_UNSUPPORTED;
  int R = 0;
  const int st = check_geometry(p, head_dim, &R);
  if (st != PA_OK) return st;
  if (!aligned(k_pages, 8) || !aligned(v_pages, 8)) return PA_ERR_ALIGN;
  SplitArgs a;
  *path = (int32_t)encode_kv_maps(&a, p, k_pages, v_pages, head_dim * elem_bytes);
  return PA_OK;
}

int pa_debug_stall_next(int64_t wait_limit_cycles) {
  if (wait_limit_cycles <= 0) return PA_ERR_SHAPE;
  g_stall_next.store(wait_limit_cycles);
  return PA_OK;
}

int pa_timing_enable(int on) {
  Timing& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  T.on = on != 0;
  return PA_OK;
}

int pa_timing_collect(int kernel, double* total_ms, int64_t* launches) {
  if (!total_ms || !launches) return PA_ERR_NULL;
  if (kernel != 0 && kernel != 1) return PA_ERR_SHAPE;
  Timing& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  double sum = 0.0;
  for (size_t i = 0; i < T.used[kernel]; ++i) {
    cudaEvent_t a = T.pool[kernel][2 * i], b = T.pool[kernel][2 * i + 1];
    if (cudaEventSynchronize(b) != cudaSuccess) return PA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return PA_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *launches = (int64_t)T.used[kernel];
  T.used[kernel] = 0;
  return PA_OK;
}

}  // extern "C"
