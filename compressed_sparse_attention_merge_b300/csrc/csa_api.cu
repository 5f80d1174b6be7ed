// C ABI of the CSA2 library: host-side validation, workspace layout, launch configuration, the device
// status word and opt-in kernel timing. Every compute step runs in the kernels of this directory; the
// host code only checks arguments and launches. Nothing here allocates device memory.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "csa_internal.cuh"

using namespace csa;

namespace {

struct DeviceInfo {
  int checked = 0;     // 0 unknown, 1 ok, -1 unsupported
  int num_sms = 0;
};
DeviceInfo g_dev[64];

// Validates the current device (sm_103) and caches its SM count.
csa_status current_device(int* num_sms) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return CSA_ERR_UNSUPPORTED_DEVICE;
  DeviceInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.num_sms = sms;
    d.checked = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (d.checked < 0) return CSA_ERR_UNSUPPORTED_DEVICE;
  if (num_sms) *num_sms = d.num_sms;
  return CSA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------------------------
// Index workspace: [header][block scores][coarse scores][kept super-blocks]
// ---------------------------------------------------------------------------------------------
struct IndexLayout {
  int64_t units, n_b_cap, n_slots, n_super, keep_super;
  size_t scores_off, coarse_off, kept_off, total;
};

IndexLayout index_layout(int64_t batch, const csa_index_args* a) {
  IndexLayout L{};
  const bool hier = (a->flags & CSA_IDX_HIER) != 0;
  L.units = batch * a->n_query;
  L.n_b_cap = ceil_div(a->max_entries, kBlockEntries);
  L.n_super = ceil_div(L.n_b_cap, kSuper);
  L.keep_super = hier ? a->keep_blocks / kSuper : 0;
  L.n_slots = hier ? (int64_t)a->keep_blocks : L.n_b_cap;
  L.scores_off = CSA_WS_HEADER_BYTES;
  L.coarse_off = round_up(L.scores_off + (size_t)L.units * L.n_slots * 4, 256);
  L.kept_off = round_up(L.coarse_off + (hier ? (size_t)L.units * L.n_super * 4 : 0), 256);
  L.total = round_up(L.kept_off + (size_t)L.units * L.keep_super * 4, 256);
  return L;
}

// ---------------------------------------------------------------------------------------------
// Attention workspace: [header][partial o][partial (m, l)]
// ---------------------------------------------------------------------------------------------
struct AttnLayout {
  int64_t units;
  int n_ct, n_wt, splits, cache_splits, win_split, last_ct;
  bool exact_prep;
  size_t o_off, ml_off, q4_off, q4sc_off, q4m_off, w4_off, w4sc_off, qh_off, total;
};

// One CTA per SM: the selected blocks of a query are cut into 128-row tiles (16 blocks) shared by the
// cache splits, and the window rows, when there are SMs to spare, get a split of their own.
AttnLayout attn_layout(int64_t batch, const csa_attn_args* a, int num_sms) {
  AttnLayout L{};
  L.units = batch * a->n_query;
  L.n_ct = (int)ceil_div(a->top_k, 16);
  L.n_wt = a->swa_rows > 0 ? (int)ceil_div(a->window, 128) : 0;
  const int64_t avail = L.units > 0 ? num_sms / L.units : 1;
  L.cache_splits = (int)(avail < 1 ? 1 : (avail < L.n_ct ? avail : L.n_ct));
  // the window tiles get a split of their own only if it still fits the one wave of CTAs
  L.win_split = (L.n_wt > 0 && L.units * (L.cache_splits + 1) <= num_sms) ? 1 : 0;
  L.splits = L.cache_splits + L.win_split;
  // When the last cache split also takes the window tiles, it gets fewer cache tiles: a window tile
  // (converted in place, its copy not overlapped with a previous tile) costs about 1.5 cache tiles.
  L.last_ct = -1;
  if (!L.win_split && L.n_wt > 0 && L.cache_splits > 1) {
    const double per = (L.n_ct + 1.5 * L.n_wt) / L.cache_splits;
    int last = (int)(per - 1.5 * L.n_wt + 0.5);
    if (last < 0) last = 0;
    if (last > L.n_ct - (L.cache_splits - 1)) last = L.n_ct - (L.cache_splits - 1);
    L.last_ct = last;
  }
  // every split writes its partial (o, m, l) to the workspace and a combine kernel merges them
  L.o_off = CSA_WS_HEADER_BYTES;
  const size_t parts = L.splits > 1 ? (size_t)L.units * L.splits * a->heads : 0;
  L.ml_off = round_up(L.o_off + parts * kLatent * 4, 256);
  // the NVFP4-query variant's rounded queries (64 head rows per unit) and window rows
  const size_t qrows = (size_t)L.units * 64;
  const size_t wrows = a->window > 0 && a->swa_rows > 0 ? (size_t)batch * a->swa_rows : 0;
  L.q4_off = round_up(L.ml_off + parts * 2 * 4, 256);
  L.q4sc_off = round_up(L.q4_off + qrows * 256, 256);
  L.q4m_off = round_up(L.q4sc_off + qrows * 32, 256);
  L.w4_off = round_up(L.q4m_off + qrows * 4, 256);
  L.w4sc_off = round_up(L.w4_off + wrows * 256, 256);
  // The exact attention's fp16 queries, converted once a query by the prepare kernel when several splits would
  // each convert them and there are enough queries for the conversions to crowd the attention's start; with a
  // few queries the extra launch costs more than it saves (measured: tiny and 1M decode lose 1-2 %, the 64K
  // decode and the 20-layer chain gain).
  L.exact_prep = L.splits > 1 && L.units >= 16;
  L.qh_off = round_up(L.w4sc_off + wrows * 32, 256);
  L.total = round_up(L.qh_off + (L.exact_prep ? qrows * kLatent * 2 : 0), 256);
  return L;
}

csa_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return CSA_ERR_ALIGNMENT;
  if (ws_bytes < need) return CSA_ERR_WORKSPACE_TOO_SMALL;
  return CSA_OK;
}

// ---------------------------------------------------------------------------------------------
// Kernel timing
// ---------------------------------------------------------------------------------------------
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<ProfRecord> recs;
  size_t max_records = 0;
  int64_t dropped = 0;
  bool pending = false;
  ProfRecord cur{};
};
Profiler g_prof;

}  // namespace

namespace csa {

// Records a timing event on s; inside stream capture the event becomes an external event node of the graph.
static cudaError_t prof_record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  e = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                          : cudaEventRecord(ev, s);
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

void prof_begin(const char* name, cudaStream_t s) {
  if (!g_prof.on) return;
  if (g_prof.recs.size() >= g_prof.max_records) { ++g_prof.dropped; g_prof.pending = false; return; }
  const size_t i = g_prof.recs.size();
  g_prof.cur = ProfRecord{name, g_prof.pool[2 * i], g_prof.pool[2 * i + 1]};
  if (prof_record(g_prof.cur.start, s) != cudaSuccess) { ++g_prof.dropped; g_prof.pending = false; return; }
  g_prof.pending = true;
}

void prof_end(cudaStream_t s) {
  if (!g_prof.on || !g_prof.pending) return;
  g_prof.pending = false;
  if (prof_record(g_prof.cur.stop, s) != cudaSuccess) { ++g_prof.dropped; return; }
  g_prof.recs.push_back(g_prof.cur);
}

cudaError_t ensure_smem_limit_fn(const void* kernel, int bytes) {
  struct Entry { const void* fn; int dev; int bytes; };
  static std::mutex mu;
  static std::vector<Entry> table;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : table)
    if (x.fn == kernel && x.dev == dev && x.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // prefer the largest shared-memory carveout, so that as many CTAs stay resident as the bytes allow
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) table.push_back(Entry{kernel, dev, bytes});
  return e;
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

thread_local char g_last_error[256] = "";

int g_fault = CSA_FAULT_NONE;
uint32_t g_fault_spin = kSpinLimit;

void debug_fault(int* fault, uint32_t* spin_limit) {
  *fault = g_fault;
  *spin_limit = g_fault == CSA_FAULT_NONE ? kSpinLimit : g_fault_spin;
}

csa_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return CSA_ERR_CUDA;
}

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

}  // namespace csa

extern "C" {

const char* csa_last_error(void) { return csa::g_last_error; }

int csa_abi_version(void) { return CSA_ABI_VERSION; }

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case CSA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
    case CSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CSA_ERR_CUDA: return "CUDA runtime error";
    case CSA_ERR_DEVICE_CHECK: return "device-side check failed (invalid index or size in device data)";
    case CSA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

size_t csa_entry_bytes(int dim) { return (dim > 0 && dim % kGroup == 0) ? (size_t)entry_bytes(dim) : 0; }
size_t csa_block_bytes(int dim) { return (dim > 0 && dim % kGroup == 0) ? (size_t)block_bytes(dim) : 0; }

csa_status csa_workspace_reset(void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  if (cudaError_t e = cudaMemsetAsync(ws, 0, CSA_WS_HEADER_BYTES, stream)) return cuda_fail(e, "workspace reset");
  return CSA_OK;
}

csa_status csa_get_device_status(void* ws, cudaStream_t stream) {
  if (ws == nullptr) return CSA_ERR_INVALID_ARG;
  uint32_t hdr[4] = {0, 0, 0, 0};
  if (cudaError_t e = cudaStreamSynchronize(stream)) return cuda_fail(e, "stream synchronize");
  if (cudaError_t e = cudaMemcpy(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost)) return cuda_fail(e, "status read");
  if (hdr[0] != 0u) {
    if (cudaError_t e = cudaMemset(ws, 0, CSA_WS_HEADER_BYTES)) return cuda_fail(e, "status clear");
  }
  switch (hdr[0]) {
    case 0: return CSA_OK;
    case CSA_ERR_TIMEOUT: return CSA_ERR_TIMEOUT;
    default: return CSA_ERR_DEVICE_CHECK;
  }
}

// ------------------------------------------------------------------------------------------------
// Host-side checks of one pack call and its kernel parameters; *empty is set when there is nothing to pack.
static csa_status pack_params(int64_t batch, const csa_pack_args* a, void* ws, PackParams* p, bool* empty) {
  if (a == nullptr || batch < 0) return CSA_ERR_INVALID_ARG;
  if (a->x_dtype != CSA_DTYPE_BF16 && a->x_dtype != CSA_DTYPE_F32) return CSA_ERR_INVALID_ARG;
  if (a->merge != 1 && a->merge != 2) return CSA_ERR_INVALID_ARG;
  if (a->scale_rule != CSA_SCALE_AMAX && a->scale_rule != CSA_SCALE_POW2) return CSA_ERR_INVALID_ARG;
  if (a->dim <= 0 || a->dim % 64 != 0 || a->dim > 1024) return CSA_ERR_INVALID_ARG;
  if (a->n_tokens < 0 || a->max_entries < 0) return CSA_ERR_INVALID_ARG;
  if (batch > 65535) return CSA_ERR_INVALID_ARG;
  const int64_t n_new = a->n_tokens / a->merge;
  *empty = batch == 0 || n_new == 0;
  if (*empty) return CSA_OK;
  if (a->x == nullptr || a->cache == nullptr) return CSA_ERR_INVALID_ARG;
  const int esz = a->x_dtype == CSA_DTYPE_BF16 ? 2 : 4;
  if (!aligned(a->x, 16) || !aligned(a->cache, 16)) return CSA_ERR_ALIGNMENT;
  if ((a->x_stride_t * esz) % 16 != 0 || (a->x_stride_b * esz) % 16 != 0 || a->cache_stride_b % 16 != 0)
    return CSA_ERR_ALIGNMENT;
  if (a->x_stride_t < a->dim) return CSA_ERR_INVALID_ARG;
  const int64_t cap_bytes = ceil_div(a->max_entries, kBlockEntries) * block_bytes(a->dim);
  if (batch > 1 && a->cache_stride_b < cap_bytes) return CSA_ERR_INVALID_ARG;
  const int64_t per_super = (int64_t)kSuper * kBlockEntries;
  const int64_t n_super = ceil_div(a->max_entries, per_super);
  if (a->coarse_sum != nullptr) {
    if (!aligned(a->coarse_sum, 16)) return CSA_ERR_ALIGNMENT;
    if (batch > 1 && a->coarse_stride_b < n_super * a->dim) return CSA_ERR_INVALID_ARG;
    if (ceil_div(n_new, per_super) + 1 > 65535) return CSA_ERR_INVALID_ARG;
  }
  *p = PackParams{};
  p->x = a->x; p->x_dtype = a->x_dtype; p->dim = a->dim; p->merge = a->merge; p->scale_rule = a->scale_rule;
  p->x_stride_b = a->x_stride_b; p->x_stride_t = a->x_stride_t; p->n_new = n_new; p->batch = batch;
  p->max_entries = a->max_entries; p->first_entry = a->first_entry;
  p->cache = a->cache; p->cache_stride_b = a->cache_stride_b;
  p->coarse_sum = a->coarse_sum; p->coarse_stride_b = a->coarse_stride_b;
  p->hdr = static_cast<uint32_t*>(ws);
  return CSA_OK;
}

csa_status csa_pack_fp4(int64_t batch, const csa_pack_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  PackParams p;
  bool empty = false;
  csa_status st = pack_params(batch, a, ws, &p, &empty);
  if (st != CSA_OK) return st;
  st = current_device(nullptr);
  if (st != CSA_OK) return st;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  if (empty) return CSA_OK;
  if (cudaError_t e = launch_pack(p, stream)) return cuda_fail(e, "pack");
  if (cudaError_t e = launch_coarse_sum(p, stream)) return cuda_fail(e, "coarse_sum");
  return CSA_OK;
}

csa_status csa_pack_fp4_multi(int n_jobs, const int64_t* batch, const csa_pack_args* args, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  if (n_jobs < 1 || n_jobs > CSA_PACK_MAX_JOBS || batch == nullptr || args == nullptr) return CSA_ERR_INVALID_ARG;
  PackParams jobs[CSA_PACK_MAX_JOBS];
  int n = 0;
  for (int j = 0; j < n_jobs; ++j) {
    bool empty = false;
    const csa_status st = pack_params(batch[j], &args[j], ws, &jobs[n], &empty);
    if (st != CSA_OK) return st;
    if (!empty) ++n;
  }
  csa_status st = current_device(nullptr);
  if (st != CSA_OK) return st;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  if (n == 0) return CSA_OK;
  if (cudaError_t e = launch_pack_multi(jobs, n, stream)) return cuda_fail(e, "pack");
  for (int j = 0; j < n; ++j)
    if (cudaError_t e = launch_coarse_sum(jobs[j], stream)) return cuda_fail(e, "coarse_sum");
  return CSA_OK;
}

csa_status csa_project_pack(int64_t batch, const csa_project_args* a, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  if (a == nullptr || batch < 0 || batch > 65535) return CSA_ERR_INVALID_ARG;
  if (a->scale_rule != CSA_SCALE_AMAX && a->scale_rule != CSA_SCALE_POW2) return CSA_ERR_INVALID_ARG;
  if (a->reserved != 0) return CSA_ERR_INVALID_ARG;
  if (a->hidden < 64 || a->hidden > 16384 || a->hidden % 64 != 0) return CSA_ERR_INVALID_ARG;
  if (a->n_tokens < 0 || a->n_tokens > (int64_t)65535 * 128 || a->max_entries < 0) return CSA_ERR_INVALID_ARG;
  const int64_t n_pairs = a->n_tokens / 2;
  const bool empty = batch == 0 || n_pairs == 0;
  if (!empty) {
    if (a->h == nullptr || a->w == nullptr || a->cache == nullptr) return CSA_ERR_INVALID_ARG;
    if (!aligned(a->h, 16) || !aligned(a->w, 16) || !aligned(a->cache, 16)) return CSA_ERR_ALIGNMENT;
    if (a->h_stride_t % 8 != 0 || a->h_stride_b % 8 != 0 || a->cache_stride_b % 16 != 0) return CSA_ERR_ALIGNMENT;
    if (a->h_stride_t < a->hidden) return CSA_ERR_INVALID_ARG;
    if (batch > 1 && a->h_stride_b < a->n_tokens * a->h_stride_t) return CSA_ERR_INVALID_ARG;
    if (batch > 1 && a->cache_stride_b < ceil_div(a->max_entries, kBlockEntries) * block_bytes(kLatent))
      return CSA_ERR_INVALID_ARG;
  }
  csa_status st = current_device(nullptr);
  if (st != CSA_OK) return st;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  if (empty) return CSA_OK;
  ProjectParams p{};
  p.h = static_cast<const __nv_bfloat16*>(a->h);
  p.h_stride_b = a->h_stride_b; p.h_stride_t = a->h_stride_t; p.hidden = a->hidden; p.n_tokens = a->n_tokens;
  p.batch = batch; p.max_entries = a->max_entries; p.cache_stride_b = a->cache_stride_b;
  p.w = static_cast<const __nv_bfloat16*>(a->w);
  p.scale_rule = a->scale_rule; p.first_entry = a->first_entry; p.cache = a->cache;
  p.hdr = static_cast<uint32_t*>(ws);
  if (cudaError_t e = launch_project_pack(p, stream)) return cuda_fail(e, "project_pack");
  return CSA_OK;
}

// ------------------------------------------------------------------------------------------------
}  // extern "C"

namespace csa {
csa_status validate_index_args(int64_t batch, const csa_index_args* a) {
  if (a == nullptr || batch < 0) return CSA_ERR_INVALID_ARG;
  if (a->n_query < 1 || a->max_entries < 0) return CSA_ERR_INVALID_ARG;
  if (a->heads != 1 && a->heads != 2 && a->heads != 4 && a->heads != 8) return CSA_ERR_INVALID_ARG;
  if (a->dim != 64 && a->dim != 128 && a->dim != 256) return CSA_ERR_INVALID_ARG;
  if (a->top_k < 1 || a->top_k > CSA_MAX_TOP_K) return CSA_ERR_INVALID_ARG;
  if ((a->flags & ~(CSA_IDX_RELU | CSA_IDX_HIER)) != 0) return CSA_ERR_INVALID_ARG;
  const bool hier = (a->flags & CSA_IDX_HIER) != 0;
  if (hier) {
    if (a->q_pos != nullptr || a->coarse_sum == nullptr) return CSA_ERR_INVALID_ARG;
    if (a->keep_blocks < kSuper || a->keep_blocks % kSuper != 0 || a->keep_blocks > 4096) return CSA_ERR_INVALID_ARG;
    if (!aligned(a->coarse_sum, 16)) return CSA_ERR_ALIGNMENT;
  }
  const int64_t units_y = hier ? batch * a->n_query : batch;
  if (units_y > 65535) return CSA_ERR_INVALID_ARG;
  if (batch == 0) return CSA_OK;
  if (a->q_idx == nullptr || a->keys == nullptr || a->n_entries == nullptr || a->out_idx == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned(a->q_idx, 16) || !aligned(a->keys, 16) || a->keys_stride_b % 16 != 0) return CSA_ERR_ALIGNMENT;
  if (batch > 1 && a->keys_stride_b < ceil_div(a->max_entries, kBlockEntries) * block_bytes(a->dim))
    return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}
}  // namespace csa

extern "C" {

size_t csa_index_topk_workspace_size(int64_t batch, const csa_index_args* a) {
  if (a == nullptr || batch < 0) return 0;
  return index_layout(batch, a).total;
}

namespace csa {
// csa_index_topk's launches, all programmatic dependents: each of its kernels waits for the kernel before it
// ahead of its first memory access.
static csa_status index_topk_run(int64_t batch, const csa_index_args* a, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  const bool early = true;
  csa_status st = validate_index_args(batch, a);
  if (st != CSA_OK) return st;
  int num_sms = 0;
  st = current_device(&num_sms);
  if (st != CSA_OK) return st;
  const IndexLayout L = index_layout(batch, a);
  st = check_ws(ws, ws_bytes, L.total);
  if (st != CSA_OK) return st;
  if (batch == 0) return CSA_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(w);
  const bool hier = (a->flags & CSA_IDX_HIER) != 0;
  const bool relu = (a->flags & CSA_IDX_RELU) != 0;
  float* scores = reinterpret_cast<float*>(w + L.scores_off);
  int32_t* kept = reinterpret_cast<int32_t*>(w + L.kept_off);

  if (hier) {
    CoarseScoreParams cp{};
    cp.q_idx = a->q_idx; cp.head_w = a->head_w; cp.n_query = a->n_query; cp.heads = a->heads; cp.dim = a->dim;
    cp.relu = relu; cp.coarse = a->coarse_sum; cp.coarse_stride_b = a->coarse_stride_b;
    cp.n_entries = a->n_entries; cp.n_super = L.n_super;
    cp.scores = reinterpret_cast<float*>(w + L.coarse_off); cp.batch = batch;
    if (cudaError_t e = launch_coarse_score(cp, stream, early)) return cuda_fail(e, "coarse_score");
    TopkParams tk{};
    tk.scores = cp.scores; tk.score_stride = L.n_super; tk.n = L.n_super; tk.k = (int)L.keep_super;
    tk.out = kept; tk.out_stride = L.keep_super; tk.units = L.units; tk.hdr = hdr;
    if (cudaError_t e = launch_topk(tk, stream, true)) return cuda_fail(e, "topk");
  }

  ScoreParams sp{};
  sp.q_idx = a->q_idx; sp.head_w = a->head_w; sp.n_query = a->n_query; sp.heads = a->heads; sp.dim = a->dim;
  sp.relu = relu; sp.keys = a->keys; sp.keys_stride_b = a->keys_stride_b; sp.n_entries = a->n_entries;
  sp.max_entries = a->max_entries; sp.q_pos = a->q_pos;
  sp.kept = hier ? kept : nullptr; sp.keep_super = (int)L.keep_super;
  sp.scores = scores; sp.score_stride = L.n_slots; sp.n_slots = L.n_slots; sp.batch = batch; sp.hdr = hdr;
  if (cudaError_t e = launch_index_score(sp, num_sms, stream, hier || early)) return cuda_fail(e, "index_score");

  TopkParams tk{};
  tk.scores = scores; tk.score_stride = L.n_slots; tk.n = L.n_slots; tk.k = a->top_k;
  tk.out = a->out_idx; tk.out_stride = a->top_k; tk.units = L.units; tk.hdr = hdr;
  if (hier) { tk.map_super = kept; tk.map_stride = (int)L.keep_super; }
  if (cudaError_t e = launch_topk(tk, stream, true)) return cuda_fail(e, "topk");

  if (a->out_block_scores != nullptr && !hier) {
    if (cudaError_t e = cudaMemcpyAsync(a->out_block_scores, scores, (size_t)L.units * L.n_slots * 4,
                                        cudaMemcpyDeviceToDevice, stream))
      return cuda_fail(e, "block score copy");
  }
  return CSA_OK;
}
}  // namespace csa

extern "C" csa_status csa_index_topk(int64_t batch, const csa_index_args* a, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  return index_topk_run(batch, a, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------------------------------
static csa_status validate_attn(int64_t batch, const csa_attn_args* a, bool prefill) {
  if (a == nullptr || batch < 0) return CSA_ERR_INVALID_ARG;
  if (a->n_query < 1 || a->max_entries < 0) return CSA_ERR_INVALID_ARG;
  if (a->heads != 16 && a->heads != 32 && a->heads != 48 && a->heads != 64) return CSA_ERR_INVALID_ARG;
  if (a->top_k < 1 || a->top_k > CSA_MAX_TOP_K) return CSA_ERR_INVALID_ARG;
  if (a->window < 0 || a->window > 1024) return CSA_ERR_INVALID_ARG;
  if (!(a->scale > 0.0f) || a->scale != a->scale) return CSA_ERR_INVALID_ARG;
  if (batch * a->n_query > 65535) return CSA_ERR_INVALID_ARG;
  if (batch == 0) return CSA_OK;
  if (a->q == nullptr || a->cache == nullptr || a->n_entries == nullptr || a->idx == nullptr || a->out == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->cache, 32) || a->cache_stride_b % 32 != 0 || !aligned(a->out, 16))
    return CSA_ERR_ALIGNMENT;
  if (batch > 1 && a->cache_stride_b < ceil_div(a->max_entries, kBlockEntries) * block_bytes(kLatent))
    return CSA_ERR_INVALID_ARG;
  if (a->window > 0) {
    if (a->swa == nullptr || a->swa_rows < 0) return CSA_ERR_INVALID_ARG;
    if (!aligned(a->swa, 16) || (a->swa_stride_b * 2) % 16 != 0) return CSA_ERR_ALIGNMENT;
    if (batch > 1 && a->swa_stride_b < a->swa_rows * kLatent) return CSA_ERR_INVALID_ARG;
    if (prefill ? a->swa_first_pos == nullptr : a->swa_len == nullptr) return CSA_ERR_INVALID_ARG;
  }
  if (prefill && a->q_pos == nullptr) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

size_t csa_sparse_attn_workspace_size(int64_t batch, const csa_attn_args* a) {
  if (a == nullptr || batch < 0) return 0;
  int num_sms = 0;
  if (current_device(&num_sms) != CSA_OK) num_sms = 148;
  return attn_layout(batch, a, num_sms).total;
}

// The attention's launches; `early` makes the attention kernel a programmatic dependent of the kernel before
// it, which is only right when that kernel belongs to the same call (the attention loads the call's queries
// and window rows before it waits).
// Which launches of the call: all of them, only the prepare kernel, or everything after it (a caller that
// launched the prepare kernel earlier on the same stream, as csa_decode_layers does).
enum AttnPhase { ATTN_ALL = 0, ATTN_PREP_ONLY = 1, ATTN_AFTER_PREP = 2 };

static csa_status sparse_attn(int64_t batch, const csa_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t stream,
                              bool prefill, bool early, bool q4 = false, int phase = ATTN_ALL) {
  csa_status st = validate_attn(batch, a, prefill);
  if (st != CSA_OK) return st;
  int num_sms = 0;
  st = current_device(&num_sms);
  if (st != CSA_OK) return st;
  const AttnLayout L = attn_layout(batch, a, num_sms);
  st = check_ws(ws, ws_bytes, L.total);
  if (st != CSA_OK) return st;
  if (batch == 0) return CSA_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  AttnParams p{};
  p.units = L.units; p.n_query = a->n_query; p.heads = a->heads;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.cache = a->cache; p.cache_stride_b = a->cache_stride_b; p.n_entries = a->n_entries;
  p.max_entries = a->max_entries; p.idx = a->idx; p.top_k = a->top_k; p.window = a->window;
  p.q_pos = prefill ? a->q_pos : nullptr;
  p.swa = static_cast<const __nv_bfloat16*>(a->swa); p.swa_stride_b = a->swa_stride_b; p.swa_rows = a->swa_rows;
  p.swa_len = a->swa_len; p.swa_first_pos = a->swa_first_pos;
  p.splits = L.splits; p.cache_splits = L.cache_splits; p.win_split = L.win_split; p.n_ct = L.n_ct; p.n_wt = L.n_wt;
  p.last_ct = L.last_ct;
  p.part_o = reinterpret_cast<float*>(w + L.o_off);
  p.part_ml = reinterpret_cast<float*>(w + L.ml_off);
  p.out = a->out; p.out_lse = a->out_lse;
  p.hdr = reinterpret_cast<uint32_t*>(w);
  p.q4 = q4 ? 1 : 0;
  debug_fault(&p.fault, &p.spin_limit);
  // The NVFP4-query variant rounds the queries and the window rows once, in a kernel of its own; the exact
  // attention converts its queries there too when many queries have several splits each (see attn_layout). The
  // attention kernel, the prepare kernel's programmatic dependent, copies the prepared operands in.
  const bool prep = q4 || L.exact_prep;
  if (prep) {
    p.q4_mult = reinterpret_cast<float*>(w + L.q4m_off);
    if (q4) {
      p.q4_codes = w + L.q4_off;
      p.q4_sc = w + L.q4sc_off;
      p.w4 = w + L.w4_off;
      p.w4_sc = w + L.w4sc_off;
    } else {
      p.qh = reinterpret_cast<__half*>(w + L.qh_off);
    }
    if (phase != ATTN_AFTER_PREP) {
      if (cudaError_t e = launch_attn_prep(p, stream, early)) return cuda_fail(e, "attn_prep");
    }
  }
  if (phase == ATTN_PREP_ONLY) return CSA_OK;
  if (cudaError_t e = launch_attn(p, stream, early || prep)) return cuda_fail(e, "attn");
  if (cudaError_t e = launch_combine(p, stream, true)) return cuda_fail(e, "combine");
  return CSA_OK;
}

csa_status csa_sparse_attn_decode(int64_t batch, const csa_attn_args* a, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  return sparse_attn(batch, a, ws, ws_bytes, stream, false, false);
}

csa_status csa_sparse_attn_prefill(int64_t batch, const csa_attn_args* a, void* ws, size_t ws_bytes,
                                   cudaStream_t stream) {
  return sparse_attn(batch, a, ws, ws_bytes, stream, true, false);
}

csa_status csa_sparse_attn_decode_nvfp4q(int64_t batch, const csa_attn_args* a, void* ws, size_t ws_bytes,
                                         cudaStream_t stream) {
  return sparse_attn(batch, a, ws, ws_bytes, stream, false, false, true);
}

csa_status csa_sparse_attn_prefill_nvfp4q(int64_t batch, const csa_attn_args* a, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
  return sparse_attn(batch, a, ws, ws_bytes, stream, true, false, true);
}

// ------------------------------------------------------------------------------------------------
csa_status csa_decode_layers(int64_t batch, int n_layers, const csa_layer_args* layers,
                             const csa_index_args* index_tmpl, const csa_attn_args* attn_tmpl, void* ws_index,
                             size_t ws_index_bytes, void* ws_attn, size_t ws_attn_bytes, cudaStream_t stream) {
  if (n_layers < 1 || layers == nullptr || index_tmpl == nullptr || attn_tmpl == nullptr || batch < 0)
    return CSA_ERR_INVALID_ARG;
  const bool causal = attn_tmpl->q_pos != nullptr;
  // every layer's calls are validated before the first launch
  int32_t* src = nullptr;
  for (int l = 0; l < n_layers; ++l) {
    const csa_layer_args& L = layers[l];
    if (L.mode != CSA_LAYER_FULL && L.mode != CSA_LAYER_REINDEX && L.mode != CSA_LAYER_REUSE) return CSA_ERR_INVALID_ARG;
    if (L.mode == CSA_LAYER_REUSE && src == nullptr) return CSA_ERR_INVALID_ARG;
    if ((L.flags & ~CSA_LAYER_ATTN_NVFP4Q) != 0) return CSA_ERR_INVALID_ARG;
    if (L.mode != CSA_LAYER_REUSE) {
      csa_index_args ia = *index_tmpl;
      ia.q_idx = L.q_idx;
      ia.out_idx = L.idx;
      ia.out_block_scores = nullptr;
      csa_status st = validate_index_args(batch, &ia);
      if (st != CSA_OK) return st;
      if (batch > 0) {
        st = check_ws(ws_index, ws_index_bytes, index_layout(batch, &ia).total);
        if (st != CSA_OK) return st;
      }
      src = L.idx;
    }
    csa_attn_args aa = *attn_tmpl;
    aa.q = L.q;
    aa.idx = src;
    aa.swa = L.swa;
    aa.out = L.out;
    aa.out_lse = L.out_lse;
    csa_status st = validate_attn(batch, &aa, causal);
    if (st != CSA_OK) return st;
  }
  src = nullptr;
  for (int l = 0; l < n_layers; ++l) {
    const csa_layer_args& L = layers[l];
    const bool q4 = (L.flags & CSA_LAYER_ATTN_NVFP4Q) != 0;
    // The layer's prepare kernel (queries and window rows, when the attention uses one) goes first: it reads
    // only the layer's inputs, so it runs beside the end of the previous layer and ahead of the indexer; the
    // attention, launched after the Top-K, implies its completion.
    {
      csa_attn_args aa = *attn_tmpl;
      aa.q = L.q;
      aa.idx = L.mode != CSA_LAYER_REUSE ? L.idx : src;
      aa.swa = L.swa;
      aa.out = L.out;
      aa.out_lse = L.out_lse;
      const csa_status st = sparse_attn(batch, &aa, ws_attn, ws_attn_bytes, stream, causal, true, q4, ATTN_PREP_ONLY);
      if (st != CSA_OK) return st;
    }
    if (L.mode != CSA_LAYER_REUSE) {
      csa_index_args ia = *index_tmpl;
      ia.q_idx = L.q_idx;
      ia.out_idx = L.idx;
      ia.out_block_scores = nullptr;
      const csa_status st = index_topk_run(batch, &ia, ws_index, ws_index_bytes, stream);
      if (st != CSA_OK) return st;
      src = L.idx;
    }
    csa_attn_args aa = *attn_tmpl;
    aa.q = L.q;
    aa.idx = src;
    aa.swa = L.swa;
    aa.out = L.out;
    aa.out_lse = L.out_lse;
    const csa_status st = sparse_attn(batch, &aa, ws_attn, ws_attn_bytes, stream, causal, true, q4, ATTN_AFTER_PREP);
    if (st != CSA_OK) return st;
  }
  return CSA_OK;
}

// ------------------------------------------------------------------------------------------------
csa_status csa_debug_set_fault(int fault, uint32_t spin_limit) {
  if (fault != CSA_FAULT_NONE && fault != CSA_FAULT_WITHHOLD_ARRIVAL) return CSA_ERR_INVALID_ARG;
  if (fault != CSA_FAULT_NONE && spin_limit == 0) return CSA_ERR_INVALID_ARG;
  csa::g_fault = fault;
  csa::g_fault_spin = spin_limit;
  return CSA_OK;
}

// ------------------------------------------------------------------------------------------------
csa_status csa_profile_begin(int max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20)) return CSA_ERR_INVALID_ARG;
  if (g_prof.on) return CSA_ERR_INVALID_ARG;
  for (auto e : g_prof.pool) cudaEventDestroy(e);
  g_prof.pool.assign(2 * (size_t)max_launches, nullptr);
  for (auto& e : g_prof.pool)
    if (cudaError_t err = cudaEventCreate(&e)) return cuda_fail(err, "cudaEventCreate");
  g_prof.recs.clear();
  g_prof.recs.reserve(max_launches);
  g_prof.max_records = max_launches;
  g_prof.dropped = 0;
  g_prof.pending = false;
  g_prof.on = true;
  return CSA_OK;
}

csa_status csa_profile_end(csa_kernel_time* out, int max_out, int* n_out, int64_t* dropped) {
  if (!g_prof.on) return CSA_ERR_INVALID_ARG;
  g_prof.on = false;
  if (cudaError_t e = cudaDeviceSynchronize()) return cuda_fail(e, "device synchronize");
  std::vector<csa_kernel_time> agg;
  for (const auto& r : g_prof.recs) {
    float ms = 0.0f;
    if (cudaError_t e = cudaEventElapsedTime(&ms, r.start, r.stop)) return cuda_fail(e, "cudaEventElapsedTime");
    size_t i = 0;
    for (; i < agg.size(); ++i)
      if (std::strncmp(agg[i].name, r.name, sizeof(agg[i].name)) == 0) break;
    if (i == agg.size()) {
      csa_kernel_time t{};
      std::strncpy(t.name, r.name, sizeof(t.name) - 1);
      agg.push_back(t);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
  }
  const int n = (int)agg.size() < max_out ? (int)agg.size() : max_out;
  for (int i = 0; i < n; ++i) out[i] = agg[i];
  if (n_out) *n_out = n;
  if (dropped) *dropped = g_prof.dropped;
  g_prof.recs.clear();
  return CSA_OK;
}

}  // extern "C"
