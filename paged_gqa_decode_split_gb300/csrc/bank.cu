// Workspace bank (pa_bank_*, declared in include/pa.h): host-side bookkeeping
// that hands out decode workspaces ("panels") for CUDA-graph capture across
// batch sizes.  No device code and no CUDA calls: device memory comes from
// the caller's allocator callback, and the device and stream are keys only.
//
// Behaviour ("DFlash2 concurrent long-context attention", section "Why the
// single-request optimization was missing from concurrent decode", and
// section "Operator validation"):
//   * a panel is shared by every batch size of one (device, stream, context
//     contract); the contract here is head_dim, num_kv_heads, num_q_heads,
//     q_len and max_ctx_len, the parameters the workspace layout depends on
//     besides the batch;
//   * a request that fits the key's current (largest) panel gets that panel,
//     so capturing batch sizes in descending order allocates once;
//   * a request that does not fit allocates a larger panel, which becomes the
//     key's current one; older panels stay allocated until the bank is
//     destroyed, because graphs captured earlier still refer to them, and every
//     pointer handed out stays valid;
//   * different streams never share a panel.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "pa.h"

struct pa_bank {
  struct Panel {
    void* ptr;
    size_t bytes;
    int32_t device;
  };
  struct Key {
    int32_t device;
    void* stream;
    int32_t head_dim, num_kv_heads, num_q_heads, q_len, max_ctx_len;
    bool operator==(const Key& o) const {
      return device == o.device && stream == o.stream && head_dim == o.head_dim && num_kv_heads == o.num_kv_heads &&
             num_q_heads == o.num_q_heads && q_len == o.q_len && max_ctx_len == o.max_ctx_len;
    }
  };
  struct Slot {
    Key key;
    size_t current;  // index into panels of the key's largest panel
  };
  pa_bank_alloc_fn alloc = nullptr;
  pa_bank_free_fn release = nullptr;
  void* user = nullptr;
  std::mutex mu;
  std::vector<Panel> panels;  // every panel ever handed out, in allocation order
  std::vector<Slot> slots;    // one per key
};

extern "C" {

pa_bank* pa_bank_create(pa_bank_alloc_fn alloc, pa_bank_free_fn release, void* user) {
  if (alloc == nullptr) return nullptr;
  pa_bank* b = new (std::nothrow) pa_bank;
  if (b == nullptr) return nullptr;
  b->alloc = alloc;
  b->release = release;
  b->user = user;
  return b;
}

int pa_bank_destroy(pa_bank* bank) {
  if (bank == nullptr) return PA_ERR_NULL;
  {
    std::lock_guard<std::mutex> lk(bank->mu);
    if (bank->release != nullptr)
      for (const pa_bank::Panel& p : bank->panels) bank->release(p.ptr, p.bytes, p.device, bank->user);
    bank->panels.clear();
    bank->slots.clear();
  }
  delete bank;
  return PA_OK;
}

int pa_bank_workspace(pa_bank* bank, const pa_params* p, int32_t device, void* stream, void** workspace,
                      size_t* workspace_bytes) {
  if (bank == nullptr || p == nullptr || workspace == nullptr || workspace_bytes == nullptr) return PA_ERR_NULL;
  if (device < 0) return PA_ERR_SHAPE;
  size_t need = 0;
  if (p->head_dim == 256) {
    need = pa_decode_fp8_workspace_bytes(p);
  } else if (p->head_dim == 128) {
    need = pa_decode_bf16_d128_workspace_bytes(p);
  } else {
    return PA_ERR_UNSUPPORTED;
  }
  if (need == 0) return PA_ERR_SHAPE;
  const pa_bank::Key key{device, stream, p->head_dim, p->num_kv_heads, p->num_q_heads, p->q_len, p->max_ctx_len};
  std::lock_guard<std::mutex> lk(bank->mu);
  pa_bank::Slot* slot = nullptr;
  for (pa_bank::Slot& s : bank->slots)
    if (s.key == key) slot = &s;
  if (slot != nullptr && bank->panels[slot->current].bytes >= need) {
    *workspace = bank->panels[slot->current].ptr;
    *workspace_bytes = bank->panels[slot->current].bytes;
    return PA_OK;
  }
  void* ptr = bank->alloc(need, device, bank->user);
  if (ptr == nullptr) return PA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ptr) % 256 != 0) {
    if (bank->release != nullptr) bank->release(ptr, need, device, bank->user);
    return PA_ERR_ALIGN;
  }
  bank->panels.push_back({ptr, need, device});
  if (slot != nullptr) {
    slot->current = bank->panels.size() - 1;
  } else {
    bank->slots.push_back({key, bank->panels.size() - 1});
  }
  *workspace = ptr;
  *workspace_bytes = need;
  return PA_OK;
}

int pa_bank_stats(pa_bank* bank, int64_t* panels, int64_t* bytes) {
  if (bank == nullptr || panels == nullptr || bytes == nullptr) return PA_ERR_NULL;
  std::lock_guard<std::mutex> lk(bank->mu);
  int64_t total = 0;
  for (const pa_bank::Panel& p : bank->panels) total += (int64_t)p.bytes;
  *panels = (int64_t)bank->panels.size();
  *bytes = total;
  return PA_OK;
}

}  // extern "C"
