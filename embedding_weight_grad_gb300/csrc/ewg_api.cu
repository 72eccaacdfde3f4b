// C ABI of the library: argument checks, workspace layout and kernel launches.
// The declarations and their contracts are in include/ewg.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "ewg.h"
#include "ewg_debug.h"
#include "ewg_internal.cuh"

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(EWG_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  // ewg_accumulate_host: the stream the grad copy runs on, and the events that order it
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t queued = nullptr, grad_in = nullptr;
};

std::mutex g_mu;
DeviceState g_devices[kMaxDevices];

// SM count of the current device; configures the kernels once per device.
int current_device(int* dev, int* num_sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(EWG_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_devices[*dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = ewg::prepare_kernels();
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    d.ready = true;
  }
  *num_sms = d.num_sms;
  return EWG_OK;
}

bool on_device(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of a foreign pointer
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

size_t elem_size(int dtype) {
  switch (dtype) {
    case EWG_INT32: return 4;
    case EWG_INT64: return 8;
    case EWG_BF16: return 2;
    case EWG_FP32: return 4;
    default: return 0;
  }
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

struct Range {
  uintptr_t lo, hi;
};

Range span(const void* p, int64_t rows, int64_t cols, int64_t row_stride, size_t es) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  const uintptr_t bytes = rows > 0 ? (static_cast<uintptr_t>(rows - 1) * row_stride + cols) * es : 0;
  return {lo, lo + bytes};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

int check_sizes(int64_t n, int64_t V, int64_t H) {
  if (n < EWG_MIN_TOKENS || n > EWG_MAX_TOKENS)
    return fail(EWG_ERR_UNSUPPORTED, "num_tokens outside [EWG_MIN_TOKENS, EWG_MAX_TOKENS]");
  if (V < 1 || V > INT32_MAX) return fail(EWG_ERR_UNSUPPORTED, "num_embeddings outside [1, 2^31)");
  if (H < 8 || H > EWG_MAX_HIDDEN || H % 8 != 0)
    return fail(EWG_ERR_UNSUPPORTED, "hidden must be a multiple of 8 in [8, EWG_MAX_HIDDEN]");
  // work items of the apply kernels are counted in 32 bits
  if (n * ((H + ewg::kCombineCols - 1) / ewg::kCombineCols) >= (int64_t(1) << 31))
    return fail(EWG_ERR_UNSUPPORTED, "num_tokens * ceil(hidden / 512) must stay below 2^31");
  return EWG_OK;
}

int check_ids(const void* ids, int ids_dtype, int dev) {
  if (ids_dtype != EWG_INT32 && ids_dtype != EWG_INT64)
    return fail(EWG_ERR_UNSUPPORTED, "ids must be int32 or int64");
  if (!ids || !aligned(ids, elem_size(ids_dtype)))
    return fail(EWG_ERR_UNSUPPORTED, "ids pointer is null or misaligned");
  if (!on_device(ids, dev)) return fail(EWG_ERR_UNSUPPORTED, "ids is not memory of the current device");
  return EWG_OK;
}

int check_mat(const void* p, int dtype, int64_t stride, int64_t H, int dev, const char* name) {
  if (dtype != EWG_BF16 && dtype != EWG_FP32)
    return fail(EWG_ERR_UNSUPPORTED, std::string(name) + " must be bf16 or fp32");
  if (!p || !aligned(p, 16)) return fail(EWG_ERR_UNSUPPORTED, std::string(name) + " is null or not 16-byte aligned");
  if (stride < H || (stride * static_cast<int64_t>(elem_size(dtype))) % 16 != 0)
    return fail(EWG_ERR_UNSUPPORTED, std::string(name) + " row stride must be >= hidden and a multiple of 16 bytes");
  if (!on_device(p, dev)) return fail(EWG_ERR_UNSUPPORTED, std::string(name) + " is not memory of the current device");
  return EWG_OK;
}

int check_all(const void* ids, int ids_dtype, int64_t n, const void* grad, int grad_dtype,
              int64_t grad_row_stride, const void* mg, int mg_dtype, int64_t V, int64_t H,
              int64_t mg_row_stride, int dev) {
  int rc = check_sizes(n, V, H);
  if (rc) return rc;
  if ((rc = check_ids(ids, ids_dtype, dev))) return rc;
  if ((rc = check_mat(grad, grad_dtype, grad_row_stride, H, dev, "grad"))) return rc;
  if ((rc = check_mat(mg, mg_dtype, mg_row_stride, H, dev, "main_grad"))) return rc;
  const Range rm = span(mg, V, H, mg_row_stride, elem_size(mg_dtype));
  if (overlap(rm, span(grad, n, H, grad_row_stride, elem_size(grad_dtype))) ||
      overlap(rm, span(ids, 1, n, n, elem_size(ids_dtype))))
    return fail(EWG_ERR_UNSUPPORTED, "main_grad overlaps grad or ids");
  return EWG_OK;
}

int check_workspace(void* ws, size_t bytes, int64_t n, int64_t H, int dev) {
  if (!ws || !aligned(ws, 256)) return fail(EWG_ERR_INVALID, "workspace is null or not 256-byte aligned");
  const size_t need = ewg::make_layout(n, H).total;
  if (bytes < need)
    return fail(EWG_ERR_INVALID, "workspace smaller than ewg_workspace_bytes(num_tokens, hidden)");
  if (!on_device(ws, dev)) return fail(EWG_ERR_INVALID, "workspace is not memory of the current device");
  return EWG_OK;
}

// The plan and apply kernels write the workspace while they read ids and grad and
// update main_grad, so none of these may share bytes with it.
int check_apart(const void* ws, int64_t n, int64_t H, Range r, const char* what) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(ws);
  if (overlap(r, {lo, lo + ewg::make_layout(n, H).total}))
    return fail(EWG_ERR_UNSUPPORTED, std::string(what) + " overlaps the workspace");
  return EWG_OK;
}

Range ids_span(const void* ids, int ids_dtype, int64_t n) { return span(ids, 1, n, n, elem_size(ids_dtype)); }

// Marks the host-side enqueue of one step in profiler timelines (a no-op without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Rows [row_begin, row_begin + rows) of the [V, H] table are kept (the whole table:
// row_begin = 0, rows = V).
int do_plan(const void* ids, int ids_dtype, int64_t n, int64_t V, int64_t row_begin,
            int64_t rows, int64_t H, void* ws, cudaStream_t stream) {
  NvtxRange range("ewg_plan");
  const ewg::Layout L = ewg::make_layout(n, H);
  const bool sharded = row_begin != 0 || rows != V;
  // a skipped id sorts as key `rows`, after the shard's own keys
  const ewg::SortPlan sp = ewg::make_sort_plan(sharded ? rows : rows - 1);
  ewg::PlanArgs a{};
  a.ids = ids;
  a.ids_int64 = ids_dtype == EWG_INT64;
  a.n = static_cast<int>(n);
  a.num_embeddings = V;
  a.row_begin = row_begin;
  a.shard_rows = rows;
  a.skip_key = sharded ? static_cast<uint32_t>(rows) : 0xffffffffu;
  a.hidden = static_cast<int>(H);
  a.id_bits = sp.id_bits;
  a.passes = sp.passes;
  a.digit_bits = sp.digit_bits;
  a.tiles = static_cast<int>(L.tiles);
  a.header = at<ewg::Header>(ws, L.header);
  a.tables = at<int>(ws, L.tables);
  a.keys_a = at<uint32_t>(ws, L.keys_a);
  a.vals_a = at<uint32_t>(ws, L.vals_a);
  a.keys_b = at<uint32_t>(ws, L.keys_b);
  a.vals_b = at<uint32_t>(ws, L.vals_b);
  a.chunks = at<int>(ws, L.chunks);
  a.chunk_cap = static_cast<int>(L.short_base + n);
  a.run_cap = static_cast<int>(ewg::max_long_runs(n));
  a.partial_cap = static_cast<int>(ewg::max_partial_rows(n));
  a.short_base = static_cast<int>(L.short_base);
  a.runs = at<int>(ws, L.runs);
  a.tile_hist = at<uint32_t>(ws, L.tile_hist);
  a.counters = at<uint32_t>(ws, L.ctl);
  a.tile_bad = at<int>(ws, L.tile_bad);
  a.list_status = at<uint32_t>(ws, L.list_status);
  a.arrivals = at<int>(ws, L.arrivals);
  cudaError_t e = ewg::launch_plan(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  return EWG_OK;
}

int do_apply(const void* grad, int grad_dtype, int64_t grad_row_stride, void* mg, int mg_dtype,
             int64_t n, int64_t V, int64_t H, int64_t mg_row_stride, void* ws, int num_sms,
             cudaStream_t stream, bool after_plan) {
  NvtxRange range("ewg_apply");
  const ewg::Layout L = ewg::make_layout(n, H);
  ewg::ApplyArgs a{};
  a.grad = grad;
  a.grad_stride = grad_row_stride;
  a.main_grad = mg;
  a.mg_stride = mg_row_stride;
  a.n = static_cast<int>(n);
  a.hidden = static_cast<int>(H);
  a.tile_cols_long = ewg::tile_cols(H, grad_dtype == EWG_BF16, true);
  a.tile_cols_rest = ewg::tile_cols(H, grad_dtype == EWG_BF16, false);
  a.num_embeddings = V;
  a.header = at<ewg::Header>(ws, L.header);
  a.tables = at<int>(ws, L.tables);
  a.chunks = at<int>(ws, L.chunks);
  a.runs = at<int>(ws, L.runs);
  a.partial = at<float>(ws, L.partial);
  a.partial_cap = static_cast<int>(ewg::max_partial_rows(n));
  a.arrivals = at<int>(ws, L.arrivals);
  a.parts = n <= ewg::kHashMaxN ? ewg::kHashParts : 1;
  // Only when the plan of the same call runs just before (and every grad row is read):
  // up to kPrefetchBytes of the first grad rows, at most half of them.
  const int64_t grad_row_bytes = H * static_cast<int64_t>(elem_size(grad_dtype));
  a.prefetch_rows =
      after_plan ? static_cast<int>(std::min<int64_t>(n / 2, ewg::kPrefetchBytes / grad_row_bytes)) : 0;
  cudaError_t e = ewg::launch_apply(a, grad_dtype == EWG_BF16, mg_dtype == EWG_BF16, num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "apply launch");
  return EWG_OK;
}

int check_shard(int64_t V, int64_t row_begin, int64_t rows) {
  if (row_begin < 0 || rows < 1 || row_begin > V - rows)
    return fail(EWG_ERR_UNSUPPORTED, "the shard [row_begin, row_begin + shard_rows) must lie in [0, num_embeddings)");
  return EWG_OK;
}

// Layout of the host-input workspace: the ordinary workspace, then the copies of ids and
// grad, each 256-byte aligned.
struct HostLayout {
  size_t ids, grad, total;
};

HostLayout host_layout(int64_t n, int64_t H, int ids_dtype, int grad_dtype) {
  HostLayout L{};
  L.ids = ewg::make_layout(n, H).total;
  L.grad = ewg::align_up(L.ids + static_cast<size_t>(n) * elem_size(ids_dtype), 256);
  L.total = ewg::align_up(L.grad + static_cast<size_t>(n) * H * elem_size(grad_dtype), 256);
  return L;
}

bool pinned_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

}  // namespace

void ewg::set_last_error(const char* msg) { g_last_error = msg; }

extern "C" {

int ewg_can_accumulate(const void* ids, int ids_dtype, int64_t num_tokens, const void* grad,
                       int grad_dtype, int64_t grad_row_stride, const void* main_grad,
                       int main_grad_dtype, int64_t num_embeddings, int64_t hidden,
                       int64_t main_grad_row_stride) {
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != EWG_OK) return 0;
  return check_all(ids, ids_dtype, num_tokens, grad, grad_dtype, grad_row_stride, main_grad,
                   main_grad_dtype, num_embeddings, hidden, main_grad_row_stride, dev) == EWG_OK;
}

size_t ewg_workspace_bytes(int64_t num_tokens, int64_t hidden) {
  if (num_tokens < 1 || num_tokens > EWG_MAX_TOKENS || hidden < 8 || hidden > EWG_MAX_HIDDEN ||
      hidden % 8 != 0)
    return 0;
  return ewg::make_layout(num_tokens, hidden).total;
}

int ewg_accumulate(const void* ids, int ids_dtype, int64_t num_tokens, const void* grad,
                   int grad_dtype, int64_t grad_row_stride, void* main_grad, int main_grad_dtype,
                   int64_t num_embeddings, int64_t hidden, int64_t main_grad_row_stride,
                   void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  rc = check_all(ids, ids_dtype, num_tokens, grad, grad_dtype, grad_row_stride, main_grad,
                 main_grad_dtype, num_embeddings, hidden, main_grad_row_stride, dev);
  if (rc) return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, num_tokens, hidden, dev))) return rc;
  if ((rc = check_apart(workspace, num_tokens, hidden, ids_span(ids, ids_dtype, num_tokens), "ids")) ||
      (rc = check_apart(workspace, num_tokens, hidden,
                        span(grad, num_tokens, hidden, grad_row_stride, elem_size(grad_dtype)), "grad")) ||
      (rc = check_apart(workspace, num_tokens, hidden,
                        span(main_grad, num_embeddings, hidden, main_grad_row_stride, elem_size(main_grad_dtype)),
                        "main_grad")))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = do_plan(ids, ids_dtype, num_tokens, num_embeddings, 0, num_embeddings, hidden, workspace, s);
  if (rc) return rc;
  return do_apply(grad, grad_dtype, grad_row_stride, main_grad, main_grad_dtype, num_tokens,
                  num_embeddings, hidden, main_grad_row_stride, workspace, sms, s, true);
}

int ewg_plan(const void* ids, int ids_dtype, int64_t num_tokens, int64_t num_embeddings,
             int64_t hidden, void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  if ((rc = check_sizes(num_tokens, num_embeddings, hidden))) return rc;
  if ((rc = check_ids(ids, ids_dtype, dev))) return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, num_tokens, hidden, dev))) return rc;
  if ((rc = check_apart(workspace, num_tokens, hidden, ids_span(ids, ids_dtype, num_tokens), "ids")))
    return rc;
  return do_plan(ids, ids_dtype, num_tokens, num_embeddings, 0, num_embeddings, hidden, workspace,
                 static_cast<cudaStream_t>(stream));
}

int ewg_apply(const void* grad, int grad_dtype, int64_t grad_row_stride, void* main_grad,
              int main_grad_dtype, int64_t num_tokens, int64_t num_embeddings, int64_t hidden,
              int64_t main_grad_row_stride, void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  if ((rc = check_sizes(num_tokens, num_embeddings, hidden))) return rc;
  if ((rc = check_mat(grad, grad_dtype, grad_row_stride, hidden, dev, "grad"))) return rc;
  if ((rc = check_mat(main_grad, main_grad_dtype, main_grad_row_stride, hidden, dev, "main_grad")))
    return rc;
  if (overlap(span(main_grad, num_embeddings, hidden, main_grad_row_stride, elem_size(main_grad_dtype)),
              span(grad, num_tokens, hidden, grad_row_stride, elem_size(grad_dtype))))
    return fail(EWG_ERR_UNSUPPORTED, "main_grad overlaps grad");
  if ((rc = check_workspace(workspace, workspace_bytes, num_tokens, hidden, dev))) return rc;
  if ((rc = check_apart(workspace, num_tokens, hidden,
                        span(grad, num_tokens, hidden, grad_row_stride, elem_size(grad_dtype)), "grad")) ||
      (rc = check_apart(workspace, num_tokens, hidden,
                        span(main_grad, num_embeddings, hidden, main_grad_row_stride, elem_size(main_grad_dtype)),
                        "main_grad")))
    return rc;
  return do_apply(grad, grad_dtype, grad_row_stride, main_grad, main_grad_dtype, num_tokens,
                  num_embeddings, hidden, main_grad_row_stride, workspace, sms,
                  static_cast<cudaStream_t>(stream), false);
}

int ewg_accumulate_shard(const void* ids, int ids_dtype, int64_t num_tokens, const void* grad,
                         int grad_dtype, int64_t grad_row_stride, void* main_grad,
                         int main_grad_dtype, int64_t num_embeddings, int64_t row_begin,
                         int64_t shard_rows, int64_t hidden, int64_t main_grad_row_stride,
                         void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  if ((rc = check_sizes(num_tokens, num_embeddings, hidden))) return rc;
  if ((rc = check_shard(num_embeddings, row_begin, shard_rows))) return rc;
  // the shard's main_grad has shard_rows rows
  rc = check_all(ids, ids_dtype, num_tokens, grad, grad_dtype, grad_row_stride, main_grad,
                 main_grad_dtype, shard_rows, hidden, main_grad_row_stride, dev);
  if (rc) return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, num_tokens, hidden, dev))) return rc;
  if ((rc = check_apart(workspace, num_tokens, hidden, ids_span(ids, ids_dtype, num_tokens), "ids")) ||
      (rc = check_apart(workspace, num_tokens, hidden,
                        span(grad, num_tokens, hidden, grad_row_stride, elem_size(grad_dtype)), "grad")) ||
      (rc = check_apart(workspace, num_tokens, hidden,
                        span(main_grad, shard_rows, hidden, main_grad_row_stride, elem_size(main_grad_dtype)),
                        "main_grad")))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = do_plan(ids, ids_dtype, num_tokens, num_embeddings, row_begin, shard_rows, hidden, workspace, s);
  if (rc) return rc;
  return do_apply(grad, grad_dtype, grad_row_stride, main_grad, main_grad_dtype, num_tokens,
                  shard_rows, hidden, main_grad_row_stride, workspace, sms, s, false);
}

int ewg_plan_shard(const void* ids, int ids_dtype, int64_t num_tokens, int64_t num_embeddings,
                   int64_t row_begin, int64_t shard_rows, int64_t hidden, void* workspace,
                   size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  if ((rc = check_sizes(num_tokens, num_embeddings, hidden))) return rc;
  if ((rc = check_shard(num_embeddings, row_begin, shard_rows))) return rc;
  if ((rc = check_ids(ids, ids_dtype, dev))) return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, num_tokens, hidden, dev))) return rc;
  if ((rc = check_apart(workspace, num_tokens, hidden, ids_span(ids, ids_dtype, num_tokens), "ids")))
    return rc;
  return do_plan(ids, ids_dtype, num_tokens, num_embeddings, row_begin, shard_rows, hidden,
                 workspace, static_cast<cudaStream_t>(stream));
}

int ewg_read_status(const void* workspace, void* stream, int* status) {
  g_last_error.clear();
  if (!workspace || !status) return fail(EWG_ERR_INVALID, "null workspace or status pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ewg::Header* h = static_cast<const ewg::Header*>(workspace);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, &h->status, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "status copy");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  *status = v;
  return EWG_OK;
}

const char* ewg_status_string(int status) {
  switch (status) {
    case EWG_OK: return "EWG_OK";
    case EWG_ERR_UNSUPPORTED: return "EWG_ERR_UNSUPPORTED";
    case EWG_ERR_INVALID: return "EWG_ERR_INVALID";
    case EWG_ERR_CUDA: return "EWG_ERR_CUDA";
    case EWG_ERR_ID_OUT_OF_RANGE: return "EWG_ERR_ID_OUT_OF_RANGE";
    case EWG_ERR_TIMEOUT: return "EWG_ERR_TIMEOUT";
    case EWG_ERR_BOUNDS: return "EWG_ERR_BOUNDS";
    default: return "EWG_ERR_UNKNOWN";
  }
}

size_t ewg_host_workspace_bytes(int64_t num_tokens, int64_t hidden, int ids_dtype,
                                int grad_dtype) {
  if (ewg_workspace_bytes(num_tokens, hidden) == 0) return 0;
  if ((ids_dtype != EWG_INT32 && ids_dtype != EWG_INT64) ||
      (grad_dtype != EWG_BF16 && grad_dtype != EWG_FP32))
    return 0;
  return host_layout(num_tokens, hidden, ids_dtype, grad_dtype).total;
}

int ewg_accumulate_host(const void* ids_host, int ids_dtype, int64_t num_tokens,
                        const void* grad_host, int grad_dtype, void* main_grad,
                        int main_grad_dtype, int64_t num_embeddings, int64_t hidden,
                        int64_t main_grad_row_stride, void* workspace, size_t workspace_bytes,
                        void* stream) {
  g_last_error.clear();
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  if ((rc = check_sizes(num_tokens, num_embeddings, hidden))) return rc;
  if (ids_dtype != EWG_INT32 && ids_dtype != EWG_INT64)
    return fail(EWG_ERR_UNSUPPORTED, "ids must be int32 or int64");
  if (grad_dtype != EWG_BF16 && grad_dtype != EWG_FP32)
    return fail(EWG_ERR_UNSUPPORTED, "grad must be bf16 or fp32");
  if (!ids_host || !grad_host || !pinned_host(ids_host) || !pinned_host(grad_host))
    return fail(EWG_ERR_UNSUPPORTED, "ids_host and grad_host must be page-locked host memory");
  if ((rc = check_mat(main_grad, main_grad_dtype, main_grad_row_stride, hidden, dev, "main_grad")))
    return rc;
  const HostLayout HL = host_layout(num_tokens, hidden, ids_dtype, grad_dtype);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < HL.total || !on_device(workspace, dev))
    return fail(EWG_ERR_INVALID, "workspace null, misaligned, not on the device or smaller than ewg_host_workspace_bytes");
  if (overlap(span(main_grad, num_embeddings, hidden, main_grad_row_stride, elem_size(main_grad_dtype)),
              {reinterpret_cast<uintptr_t>(workspace), reinterpret_cast<uintptr_t>(workspace) + HL.total}))
    return fail(EWG_ERR_UNSUPPORTED, "main_grad overlaps the workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t ids_bytes = static_cast<size_t>(num_tokens) * elem_size(ids_dtype);
  const size_t grad_bytes = static_cast<size_t>(num_tokens) * hidden * elem_size(grad_dtype);

  std::lock_guard<std::mutex> lock(g_mu);   // the copy stream and events are shared
  DeviceState& d = g_devices[dev];
  cudaError_t e = cudaSuccess;
  if (!d.copy_stream) {
    e = cudaStreamCreateWithFlags(&d.copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.queued, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.grad_in, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "copy stream set-up");
  }
  // The grad copy starts after the work already queued on `stream` (an earlier call may
  // still read this workspace) and overlaps the ids copy and the plan.
  e = cudaEventRecord(d.queued, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d.copy_stream, d.queued, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + HL.grad, grad_host, grad_bytes, cudaMemcpyHostToDevice, d.copy_stream);
  if (e == cudaSuccess) e = cudaEventRecord(d.grad_in, d.copy_stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + HL.ids, ids_host, ids_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "host input copies");
  rc = do_plan(ws + HL.ids, ids_dtype, num_tokens, num_embeddings, 0, num_embeddings, hidden, workspace, s);
  if (rc) return rc;
  e = cudaStreamWaitEvent(s, d.grad_in, 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  return do_apply(ws + HL.grad, grad_dtype, hidden, main_grad, main_grad_dtype, num_tokens,
                  num_embeddings, hidden, main_grad_row_stride, workspace, sms, s, false);
}

const char* ewg_last_error(void) { return g_last_error.c_str(); }

#ifdef EWG_DEBUG
int ewg_debug_lookback_probe(void* words, int tile, int poll_limit, int* out, void* stream) {
  g_last_error.clear();
  if (!words || !out || tile < 1 || poll_limit < 1)
    return fail(EWG_ERR_INVALID, "null pointer, tile < 1 or poll_limit < 1");
  cudaError_t e = ewg::launch_lookback_probe(static_cast<uint32_t*>(words), tile, poll_limit, out,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "look-back probe launch");
  return EWG_OK;
}
#endif

int ewg_version(void) { return 1; }

}  // extern "C"
