// The C ABI declared in include/ep_gb300.h: argument validation (all on the
// host, before any CUDA call, so invalid calls fail synchronously and never
// reach the GPU), per-device property cache, status strings and the
// per-thread detail message.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ep_internal.h"

namespace ep {

namespace {

thread_local char g_last_error[512] = "";

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

void clear_error() { g_last_error[0] = '\0'; }

ep_status_t fail(ep_status_t status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

ep_status_t cuda_fail(cudaError_t err, const char *what) {
  return fail(EP_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

const DeviceInfo *current_device_info() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fail(EP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_dev_mu);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    int major = 0, minor = 0, sms = 0, optin = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess) {
      cuda_fail(e, "cudaDeviceGetAttribute");
      return nullptr;
    }
    if (major != 10 || minor != 3) {
      fail(EP_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
           minor);
      return nullptr;
    }
    d.num_sms = sms;
    d.max_smem_per_block_optin = (size_t)optin;
    d.smem_per_sm = (size_t)per_sm;
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  return &g_dev[dev];
}

ep_status_t check_routing_sizes(const char *fn, int num_topk, int num_experts, int num_ranks) {
  if (num_topk < 1 || num_topk > EP_MAX_TOPK)
    return fail(num_topk < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_topk=%d not in [1, %d]", fn,
                num_topk, EP_MAX_TOPK);
  if (num_ranks < 1 || num_ranks > EP_MAX_RANKS)
    return fail(num_ranks < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_ranks=%d not in [1, %d]", fn,
                num_ranks, EP_MAX_RANKS);
  if (num_experts < num_ranks || num_experts > EP_MAX_EXPERTS)
    return fail(num_experts < num_ranks ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED,
                "%s: num_experts=%d not in [num_ranks=%d, %d]", fn, num_experts, num_ranks, EP_MAX_EXPERTS);
  if (num_experts % num_ranks != 0)
    return fail(EP_ERR_INVALID_ARG, "%s: num_experts=%d is not a multiple of num_ranks=%d", fn, num_experts,
                num_ranks);
  return EP_OK;
}

ep_status_t check_ptr(const char *fn, const char *name, const void *p, size_t align, bool required) {
  if (p == nullptr) {
    if (required) return fail(EP_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
    return EP_OK;
  }
  if (!aligned(p, align)) return fail(EP_ERR_INVALID_ARG, "%s: %s is not %zu-byte aligned", fn, name, align);
  return EP_OK;
}

namespace {

#define EP_CHECK(expr)                   \
  do {                                   \
    const ep_status_t _s = (expr);       \
    if (_s != EP_OK) return _s;          \
  } while (0)

// Validates the arguments of a rank-path dispatch (host only) and fills `a`.
ep_status_t dispatch_args(const char *fn, const ep_dispatch_args_t *args, DispatchArgs &a) {
  if (args == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: args is NULL", fn);
  const ep_dispatch_args_t &x = *args;
  if (x.num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, x.num_tokens);
  if (x.dtype != EP_DTYPE_BF16 && x.dtype != EP_DTYPE_FP8_E4M3 && x.dtype != EP_DTYPE_FP8_E4M3_PACKED)
    return fail(EP_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)x.dtype);
  const bool fp8 = x.dtype != EP_DTYPE_BF16;
  const bool packed = x.dtype == EP_DTYPE_FP8_E4M3_PACKED;
  if (x.hidden < 1) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d < 1", fn, x.hidden);
  if (x.hidden > EP_MAX_HIDDEN)
    return fail(EP_ERR_UNSUPPORTED, "%s: hidden=%d > %d", fn, x.hidden, EP_MAX_HIDDEN);
  if (x.hidden % (fp8 ? EP_FP8_GROUP : 8) != 0)
    return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d is not a multiple of %d", fn, x.hidden,
                fp8 ? EP_FP8_GROUP : 8);
  EP_CHECK(check_routing_sizes(fn, x.num_topk, x.num_experts, x.num_ranks));
  if (x.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "%s: recv_capacity=%d < 0", fn, x.recv_capacity);
  const bool any = x.num_tokens > 0;
  const bool rows = x.recv_capacity > 0;
  EP_CHECK(check_ptr(fn, "x", x.x, 16, any));
  EP_CHECK(check_ptr(fn, "topk_idx", x.topk_idx, 8, any));
  if (x.layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.token_slot", x.layout->token_slot, 4, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", x.layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", x.layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "recv_x", x.recv_x, 16, rows));
  EP_CHECK(check_ptr(fn, "recv_x_scales", x.recv_x_scales, 4, fp8 && !packed && rows));
  EP_CHECK(check_ptr(fn, "recv_src_idx", x.recv_src_idx, 4, false));
  EP_CHECK(check_ptr(fn, "recv_topk_idx", x.recv_topk_idx, 4, false));
  EP_CHECK(check_ptr(fn, "recv_topk_weights", x.recv_topk_weights, 4, false));
  EP_CHECK(check_ptr(fn, "topk_weights", x.topk_weights, 4, any && x.recv_topk_weights != nullptr));
  EP_CHECK(check_ptr(fn, "cumulative_recv_stats", x.cumulative_recv_stats, 4, false));
  a.x = static_cast<const uint16_t *>(x.x);
  a.num_tokens = x.num_tokens;
  a.hidden = x.hidden;
  a.num_topk = x.num_topk;
  a.num_experts = x.num_experts;
  a.num_ranks = x.num_ranks;
  a.topk_idx = x.topk_idx;
  a.topk_weights = x.topk_weights;
  a.token_slot = x.layout->token_slot;
  a.error_word = x.layout->error_word;
  a.expanded = false;
  a.expert_offset = nullptr;
  a.num_rows_per_expert = nullptr;
  a.zero_padding = false;
  a.fp8 = fp8;
  a.packed_row_bytes = packed ? (int)fp8_packed_row_bytes(x.hidden) : 0;
  a.work_counters = x.layout->work_counters;  // words 0-1: dispatch
  a.recv_x = x.recv_x;
  a.recv_x_scales = packed ? nullptr : x.recv_x_scales;
  a.recv_src_idx = x.recv_src_idx;
  a.recv_topk_idx = x.recv_topk_idx;
  a.recv_topk_weights = x.recv_topk_weights;
  a.recv_capacity = x.recv_capacity;
  a.recv_stats = x.cumulative_recv_stats;
  return EP_OK;
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" {

size_t ep_layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks) {
  if (num_tokens < 0 || num_ranks < 1 || num_ranks > EP_MAX_RANKS) return 0;
  return layout_workspace_bytes(num_tokens, num_experts, num_ranks);
}

ep_status_t ep_get_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, const ep_layout_t *layout, void *workspace, size_t workspace_bytes,
                          ep_stream_t stream) {
  static const char *fn = "ep_get_layout";
  clear_error();
  if (num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, num_tokens);
  EP_CHECK(check_routing_sizes(fn, num_topk, num_experts, num_ranks));
  const bool any = num_tokens > 0;
  EP_CHECK(check_ptr(fn, "topk_idx", topk_idx, 8, any));
  if (layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.num_tokens_per_expert", layout->num_tokens_per_expert, 4, true));
  EP_CHECK(check_ptr(fn, "layout.num_tokens_per_rank", layout->num_tokens_per_rank, 4, true));
  EP_CHECK(check_ptr(fn, "layout.rank_prefix", layout->rank_prefix, 4, true));
  EP_CHECK(check_ptr(fn, "layout.is_token_in_rank", layout->is_token_in_rank, 16, any));
  EP_CHECK(check_ptr(fn, "layout.token_slot", layout->token_slot, 16, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "workspace", workspace, 16, true));
  const size_t need = layout_workspace_bytes(num_tokens, num_experts, num_ranks);
  if (workspace_bytes < need)
    return fail(EP_ERR_INVALID_ARG, "%s: workspace_bytes=%zu < %zu needed", fn, workspace_bytes, need);
  return launch_layout(topk_idx, num_tokens, num_topk, num_experts, num_ranks, *layout, workspace,
                       reinterpret_cast<cudaStream_t>(stream));
}

size_t ep_fp8_packed_row_bytes(int hidden) {
  if (hidden < EP_FP8_GROUP || hidden % EP_FP8_GROUP != 0 || hidden > EP_MAX_HIDDEN) return 0;
  return fp8_packed_row_bytes(hidden);
}

ep_status_t ep_dispatch_ex(const ep_dispatch_args_t *args, ep_stream_t stream) {
  clear_error();
  DispatchArgs a;
  EP_CHECK(dispatch_args("ep_dispatch", args, a));
  return launch_dispatch(a, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_get_layout_and_dispatch(const ep_dispatch_args_t *args, void *workspace, size_t workspace_bytes,
                                       ep_stream_t stream) {
  static const char *fn = "ep_get_layout_and_dispatch";
  clear_error();
  DispatchArgs a;
  EP_CHECK(dispatch_args(fn, args, a));
  const ep_layout_t *layout = args->layout;
  const bool any = a.num_tokens > 0;
  EP_CHECK(check_ptr(fn, "layout.num_tokens_per_expert", layout->num_tokens_per_expert, 4, true));
  EP_CHECK(check_ptr(fn, "layout.num_tokens_per_rank", layout->num_tokens_per_rank, 4, true));
  EP_CHECK(check_ptr(fn, "layout.rank_prefix", layout->rank_prefix, 4, true));
  EP_CHECK(check_ptr(fn, "layout.is_token_in_rank", layout->is_token_in_rank, 16, any));
  EP_CHECK(check_ptr(fn, "layout.token_slot", layout->token_slot, 16, any));
  EP_CHECK(check_ptr(fn, "workspace", workspace, 16, true));
  const size_t need = layout_workspace_bytes(a.num_tokens, a.num_experts, a.num_ranks);
  if (workspace_bytes < need)
    return fail(EP_ERR_INVALID_ARG, "%s: workspace_bytes=%zu < %zu needed", fn, workspace_bytes, need);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((a.fp8 || kBf16WarpSpecialised) && a.num_tokens > 0 && a.num_tokens <= local_layout_max_tokens()) {
    // One layout launch; the dispatch finishes the slots (adds each block's
    // base, writes them back) and counts the experts as it moves the rows.
    const int32_t *local_base = nullptr;
    int table_blocks = 0;
    EP_CHECK(launch_layout_local(args->topk_idx, a.num_tokens, a.num_topk, a.num_experts, a.num_ranks, *layout,
                                 workspace, s, &local_base, &table_blocks));
    a.local_base = local_base;
    a.local_table_blocks = table_blocks;
    a.token_slot_out = layout->token_slot;
    a.num_tokens_per_expert = layout->num_tokens_per_expert;
    a.rank_prefix = layout->rank_prefix;
    a.num_tokens_per_rank = layout->num_tokens_per_rank;
  } else {
    EP_CHECK(launch_layout(args->topk_idx, a.num_tokens, a.num_topk, a.num_experts, a.num_ranks, *layout, workspace,
                           s));
  }
  // The kernel ahead of the dispatch is the layout, which writes nothing the
  // dispatch reads before its wait; so its first rows load and cast early.
  a.early_rows = kEarlyRows;
  return launch_dispatch(a, s);
}

ep_status_t ep_dispatch(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                        const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                        const ep_layout_t *layout, ep_dtype_t dtype, void *recv_x, float *recv_x_scales,
                        int32_t *recv_src_idx, int32_t *recv_topk_idx, float *recv_topk_weights,
                        int recv_capacity, ep_stream_t stream) {
  const ep_dispatch_args_t a = {x,      num_tokens,   hidden,        topk_idx,      topk_weights,
                                num_topk, num_experts, num_ranks,    layout,        dtype,
                                recv_x, recv_x_scales, recv_src_idx, recv_topk_idx, recv_topk_weights,
                                recv_capacity, nullptr};
  return ep_dispatch_ex(&a, stream);
}

ep_status_t ep_combine_ex(const ep_combine_args_t *args, ep_stream_t stream) {
  static const char *fn = "ep_combine";
  clear_error();
  if (args == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: args is NULL", fn);
  const ep_combine_args_t &x = *args;
  if (x.num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, x.num_tokens);
  if (x.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "%s: recv_capacity=%d < 0", fn, x.recv_capacity);
  if (x.hidden < 1) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d < 1", fn, x.hidden);
  if (x.hidden > EP_MAX_HIDDEN)
    return fail(EP_ERR_UNSUPPORTED, "%s: hidden=%d > %d", fn, x.hidden, EP_MAX_HIDDEN);
  if (x.hidden % 8 != 0) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d is not a multiple of 8", fn, x.hidden);
  if (x.num_ranks < 1 || x.num_ranks > EP_MAX_RANKS)
    return fail(x.num_ranks < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_ranks=%d not in [1, %d]",
                fn, x.num_ranks, EP_MAX_RANKS);
  const bool weighted = x.topk_weights != nullptr;
  if ((x.topk_idx == nullptr) != (x.topk_weights == nullptr))
    return fail(EP_ERR_INVALID_ARG, "%s: topk_idx and topk_weights must both be given or both be NULL", fn);
  const bool any = x.num_tokens > 0;
  if (weighted) {
    EP_CHECK(check_routing_sizes(fn, x.num_topk, x.num_experts, x.num_ranks));
    EP_CHECK(check_ptr(fn, "topk_idx", x.topk_idx, 8, any));
    EP_CHECK(check_ptr(fn, "topk_weights", x.topk_weights, 4, any));
  }
  EP_CHECK(check_ptr(fn, "y", x.y, 16, x.recv_capacity > 0 && any));
  if (x.layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.token_slot", x.layout->token_slot, 4, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", x.layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", x.layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "out", x.out, 16, any));
  EP_CHECK(check_ptr(fn, "bias0", x.bias0, 16, false));
  EP_CHECK(check_ptr(fn, "bias1", x.bias1, 16, false));
  CombineArgs a;
  a.y = static_cast<const uint16_t *>(x.y);
  a.recv_capacity = x.recv_capacity;
  a.hidden = x.hidden;
  a.num_tokens = x.num_tokens;
  a.num_ranks = x.num_ranks;
  a.expanded = false;
  a.num_topk = weighted ? x.num_topk : 0;
  a.num_experts = weighted ? x.num_experts : x.num_ranks;
  a.token_slot = x.layout->token_slot;
  a.error_word = x.layout->error_word;
  a.topk_idx = x.topk_idx;
  a.topk_weights = x.topk_weights;
  a.bias0 = static_cast<const uint16_t *>(x.bias0);
  a.bias1 = static_cast<const uint16_t *>(x.bias1);
  a.out = static_cast<uint16_t *>(x.out);
  a.work_counters = x.layout->work_counters != nullptr ? x.layout->work_counters + 2 : nullptr;  // words 2-3: combine
  return launch_combine(a, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_combine(const void *y, int recv_capacity, int hidden, const ep_layout_t *layout,
                       int num_tokens, int num_ranks, const int64_t *topk_idx, const float *topk_weights,
                       int num_topk, int num_experts, void *out, ep_stream_t stream) {
  const ep_combine_args_t a = {y,        recv_capacity, hidden,       layout,  num_tokens, num_ranks, topk_idx,
                               topk_weights, num_topk,  num_experts,  nullptr, nullptr,    out};
  return ep_combine_ex(&a, stream);
}

size_t ep_expanded_layout_workspace_bytes(int num_tokens, int num_experts) {
  if (num_tokens < 0 || num_experts < 1 || num_experts > EP_MAX_EXPERTS) return 0;
  return expanded_layout_workspace_bytes(num_tokens, num_experts);
}

ep_status_t ep_get_layout_expanded(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                   int expert_alignment, const ep_expanded_layout_t *layout, void *workspace,
                                   size_t workspace_bytes, ep_stream_t stream) {
  static const char *fn = "ep_get_layout_expanded";
  clear_error();
  if (num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, num_tokens);
  if (num_topk < 1 || num_topk > EP_MAX_TOPK)
    return fail(num_topk < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_topk=%d not in [1, %d]", fn,
                num_topk, EP_MAX_TOPK);
  if (num_experts < 1 || num_experts > EP_MAX_EXPERTS)
    return fail(num_experts < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_experts=%d not in [1, %d]",
                fn, num_experts, EP_MAX_EXPERTS);
  if (expert_alignment < 1 || expert_alignment > 4096)
    return fail(EP_ERR_INVALID_ARG, "%s: expert_alignment=%d not in [1, 4096]", fn, expert_alignment);
  const bool any = num_tokens > 0;
  EP_CHECK(check_ptr(fn, "topk_idx", topk_idx, 8, any));
  if (layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.num_rows_per_expert", layout->num_rows_per_expert, 4, true));
  EP_CHECK(check_ptr(fn, "layout.expert_offset", layout->expert_offset, 4, true));
  EP_CHECK(check_ptr(fn, "layout.token_slot", layout->token_slot, 16, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "workspace", workspace, 16, true));
  const size_t need = expanded_layout_workspace_bytes(num_tokens, num_experts);
  if (workspace_bytes < need)
    return fail(EP_ERR_INVALID_ARG, "%s: workspace_bytes=%zu < %zu needed", fn, workspace_bytes, need);
  return launch_layout_expanded(topk_idx, num_tokens, num_topk, num_experts, expert_alignment, *layout,
                                workspace, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_dispatch_expanded(const ep_dispatch_expanded_args_t *args, ep_stream_t stream) {
  static const char *fn = "ep_dispatch_expanded";
  clear_error();
  if (args == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: args is NULL", fn);
  const ep_dispatch_expanded_args_t &x = *args;
  if (x.num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, x.num_tokens);
  if (x.dtype != EP_DTYPE_BF16 && x.dtype != EP_DTYPE_FP8_E4M3 && x.dtype != EP_DTYPE_FP8_E4M3_PACKED)
    return fail(EP_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)x.dtype);
  const bool fp8 = x.dtype != EP_DTYPE_BF16;
  const bool packed = x.dtype == EP_DTYPE_FP8_E4M3_PACKED;
  if (x.hidden < 1) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d < 1", fn, x.hidden);
  if (x.hidden > EP_MAX_HIDDEN)
    return fail(EP_ERR_UNSUPPORTED, "%s: hidden=%d > %d", fn, x.hidden, EP_MAX_HIDDEN);
  if (x.hidden % (fp8 ? EP_FP8_GROUP : 8) != 0)
    return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d is not a multiple of %d", fn, x.hidden,
                fp8 ? EP_FP8_GROUP : 8);
  EP_CHECK(check_routing_sizes(fn, x.num_topk, x.num_experts, x.num_ranks));
  if (x.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "%s: recv_capacity=%d < 0", fn, x.recv_capacity);
  const bool any = x.num_tokens > 0;
  const bool rows = x.recv_capacity > 0;
  EP_CHECK(check_ptr(fn, "x", x.x, 16, any));
  EP_CHECK(check_ptr(fn, "topk_idx", x.topk_idx, 8, any));
  if (x.layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.token_slot", x.layout->token_slot, 4, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", x.layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", x.layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "layout.expert_offset", x.layout->expert_offset, 4, x.zero_padding != 0));
  EP_CHECK(check_ptr(fn, "layout.num_rows_per_expert", x.layout->num_rows_per_expert, 4, x.zero_padding != 0));
  EP_CHECK(check_ptr(fn, "recv_x", x.recv_x, 16, rows));
  EP_CHECK(check_ptr(fn, "recv_x_scales", x.recv_x_scales, 4, fp8 && !packed && rows));
  EP_CHECK(check_ptr(fn, "recv_src_idx", x.recv_src_idx, 4, false));
  EP_CHECK(check_ptr(fn, "recv_topk_idx", x.recv_topk_idx, 4, false));
  EP_CHECK(check_ptr(fn, "recv_topk_weights", x.recv_topk_weights, 4, false));
  EP_CHECK(check_ptr(fn, "topk_weights", x.topk_weights, 4, any && x.recv_topk_weights != nullptr));
  EP_CHECK(check_ptr(fn, "cumulative_recv_stats", x.cumulative_recv_stats, 4, false));
  DispatchArgs a;
  a.x = static_cast<const uint16_t *>(x.x);
  a.num_tokens = x.num_tokens;
  a.hidden = x.hidden;
  a.num_topk = x.num_topk;
  a.num_experts = x.num_experts;
  a.num_ranks = x.num_ranks;
  a.topk_idx = x.topk_idx;
  a.topk_weights = x.topk_weights;
  a.token_slot = x.layout->token_slot;
  a.error_word = x.layout->error_word;
  a.expanded = true;
  a.expert_offset = x.layout->expert_offset;
  a.num_rows_per_expert = x.layout->num_rows_per_expert;
  a.zero_padding = x.zero_padding != 0;
  a.fp8 = fp8;
  a.packed_row_bytes = packed ? (int)fp8_packed_row_bytes(x.hidden) : 0;
  a.work_counters = x.layout->work_counters;  // words 0-1: dispatch
  a.recv_x = x.recv_x;
  a.recv_x_scales = packed ? nullptr : x.recv_x_scales;
  a.recv_src_idx = x.recv_src_idx;
  a.recv_topk_idx = x.recv_topk_idx;
  a.recv_topk_weights = x.recv_topk_weights;
  a.recv_capacity = x.recv_capacity;
  a.recv_stats = x.cumulative_recv_stats;
  return launch_dispatch(a, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_combine_expanded(const ep_combine_expanded_args_t *args, ep_stream_t stream) {
  static const char *fn = "ep_combine_expanded";
  clear_error();
  if (args == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: args is NULL", fn);
  const ep_combine_expanded_args_t &x = *args;
  if (x.num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, x.num_tokens);
  if (x.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "%s: recv_capacity=%d < 0", fn, x.recv_capacity);
  if (x.hidden < 1) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d < 1", fn, x.hidden);
  if (x.hidden > EP_MAX_HIDDEN)
    return fail(EP_ERR_UNSUPPORTED, "%s: hidden=%d > %d", fn, x.hidden, EP_MAX_HIDDEN);
  if (x.hidden % 8 != 0) return fail(EP_ERR_INVALID_ARG, "%s: hidden=%d is not a multiple of 8", fn, x.hidden);
  if (x.num_topk < 1 || x.num_topk > EP_MAX_TOPK)
    return fail(x.num_topk < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_topk=%d not in [1, %d]", fn,
                x.num_topk, EP_MAX_TOPK);
  const bool weighted = x.topk_weights != nullptr;
  if ((x.topk_idx == nullptr) != (x.topk_weights == nullptr))
    return fail(EP_ERR_INVALID_ARG, "%s: topk_idx and topk_weights must both be given or both be NULL", fn);
  const bool any = x.num_tokens > 0;
  if (weighted) {
    if (x.num_experts < 1 || x.num_experts > EP_MAX_EXPERTS)
      return fail(EP_ERR_INVALID_ARG, "%s: num_experts=%d not in [1, %d]", fn, x.num_experts, EP_MAX_EXPERTS);
    EP_CHECK(check_ptr(fn, "topk_idx", x.topk_idx, 8, any));
    EP_CHECK(check_ptr(fn, "topk_weights", x.topk_weights, 4, any));
  }
  EP_CHECK(check_ptr(fn, "y", x.y, 16, x.recv_capacity > 0 && any));
  if (x.layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  EP_CHECK(check_ptr(fn, "layout.token_slot", x.layout->token_slot, 4, any));
  EP_CHECK(check_ptr(fn, "layout.error_word", x.layout->error_word, 4, true));
  EP_CHECK(check_ptr(fn, "layout.work_counters", x.layout->work_counters, 16, false));
  EP_CHECK(check_ptr(fn, "out", x.out, 16, any));
  EP_CHECK(check_ptr(fn, "bias0", x.bias0, 16, false));
  EP_CHECK(check_ptr(fn, "bias1", x.bias1, 16, false));
  CombineArgs a;
  a.y = static_cast<const uint16_t *>(x.y);
  a.recv_capacity = x.recv_capacity;
  a.hidden = x.hidden;
  a.num_tokens = x.num_tokens;
  a.num_ranks = 1;  // unused by the expanded reduce
  a.expanded = true;
  a.num_topk = x.num_topk;
  a.num_experts = weighted ? x.num_experts : 1;
  a.token_slot = x.layout->token_slot;
  a.error_word = x.layout->error_word;
  a.topk_idx = x.topk_idx;
  a.topk_weights = x.topk_weights;
  a.bias0 = static_cast<const uint16_t *>(x.bias0);
  a.bias1 = static_cast<const uint16_t *>(x.bias1);
  a.out = static_cast<uint16_t *>(x.out);
  a.work_counters = x.layout->work_counters != nullptr ? x.layout->work_counters + 2 : nullptr;  // words 2-3: combine
  return launch_combine(a, reinterpret_cast<cudaStream_t>(stream));
}

const char *ep_status_str(ep_status_t status) {
  switch (status) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
  }
  return "EP_STATUS_UNKNOWN";
}

const char *ep_last_error(void) { return g_last_error; }

int ep_abi_version(void) { return EP_ABI_VERSION; }

}  // extern "C"
