// C ABI of libw4a16.so: argument validation and dispatch (include/w4a16.h).
//
// Every check here runs on the host before any CUDA call, so a bad argument is
// reported even on a machine without a GPU, and nothing is launched on error.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "w4a16_internal.h"

namespace w4 {
namespace {

constexpr int MAX_DIM = 1 << 20;
constexpr int MAX_DEVICES = 64;
constexpr int MAX_ACT_ORDER_GROUPS = 8192;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool valid_group(int group) { return group == -1 || group == 32 || group == 64 || group == 128; }

int resolve_group(int group, int K) { return group == -1 ? K : group; }

w4_status check_dims(int K, int N, int group, int dtype) {
  if (K < 1 || N < 1 || K > MAX_DIM || N > MAX_DIM) return W4_ERR_SHAPE;
  if (!valid_group(group)) return W4_ERR_GROUP;
  if (K % resolve_group(group, K) != 0) return W4_ERR_GROUP;
  if (dtype != W4_F16 && dtype != W4_BF16) return W4_ERR_DTYPE;
  return W4_OK;
}

w4_status check_layout_dims(int K, int N, int layout) {
  if (layout == W4_LAYOUT_STD) {
    if (K % 8 || N % 8) return W4_ERR_SHAPE;
  } else if (layout == W4_LAYOUT_TILE) {
    if (K % 64 || N % 16) return W4_ERR_SHAPE;
  } else {
    return W4_ERR_LAYOUT;
  }
  return W4_OK;
}

struct CachedInfo {
  bool valid = false;
  DeviceInfo info{};
};
CachedInfo g_info[MAX_DEVICES];
std::mutex g_info_mu;

// The current device must be compute capability 10.3 (the kernels are sm_103a only).
w4_status check_arch() {
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return W4_ERR_CUDA;
  if (info.major != 10 || info.minor != 3) return W4_ERR_ARCH;
  return W4_OK;
}

// The last CUDA error an entry point reported on this thread (w4_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// The GEMM entry points' implementation (defined below the C ABI).
w4_status gemm_impl(const void* x, const int32_t* qw, const void* scales, const int32_t* zeros,
                    const int32_t* perm, const void* bias, void* y, int M, int N, int K,
                    int group, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                    int test_stall);

w4_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return W4_OK;
  g_last_cuda_error = e;
  return W4_ERR_CUDA;
}

}  // namespace

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_info_mu);
  if (!g_info[dev].valid) {
    DeviceInfo d{};
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                    dev)) != cudaSuccess)
      return e;
    g_info[dev].info = d;
    g_info[dev].valid = true;
  }
  *out = g_info[dev].info;
  return cudaSuccess;
}

}  // namespace w4

using namespace w4;

extern "C" {

const char* w4_status_string(w4_status s) {
  switch (s) {
    case W4_OK: return "W4_OK";
    case W4_ERR_NULL: return "W4_ERR_NULL: a required pointer is NULL";
    case W4_ERR_SHAPE: return "W4_ERR_SHAPE: M, K or N out of range or not a multiple the layout needs";
    case W4_ERR_GROUP: return "W4_ERR_GROUP: group must be 32, 64, 128 or -1 and divide K";
    case W4_ERR_ALIGN: return "W4_ERR_ALIGN: a pointer is not 16-byte aligned";
    case W4_ERR_DTYPE: return "W4_ERR_DTYPE: dtype must be W4_F16 or W4_BF16";
    case W4_ERR_LAYOUT: return "W4_ERR_LAYOUT: layout must be W4_LAYOUT_STD or W4_LAYOUT_TILE";
    case W4_ERR_ALIAS: return "W4_ERR_ALIAS: an output overlaps an input";
    case W4_ERR_ARCH: return "W4_ERR_ARCH: the current device is not compute capability 10.3";
    case W4_ERR_CUDA: return "W4_ERR_CUDA: a CUDA call or kernel launch failed";
    case W4_ERR_WORKSPACE: return "W4_ERR_WORKSPACE: workspace missing or too small";
    case W4_ERR_GIDX: return "W4_ERR_GIDX: g_idx out of range or groups not of equal size";
    case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT: a kernel gave up on a pipeline wait";
    case W4_ERR_EXPERT_ROWS:
      return "W4_ERR_EXPERT_ROWS: an expert's rows were invalid or more than max_rows_per_expert";
    default: return "unknown w4_status";
  }
}

const char* w4_last_cuda_error(void) {
  static thread_local char buf[256];
  if (g_last_cuda_error == cudaSuccess) return "no CUDA error";
  snprintf(buf, sizeof(buf), "%s: %s", cudaGetErrorName(g_last_cuda_error),
           cudaGetErrorString(g_last_cuda_error));
  return buf;
}

int w4_abi_version(void) { return 2; }

w4_status w4_repack_sizes(int K, int N, int group, int layout, size_t* qw_bytes,
                          size_t* zeros_bytes, size_t* scales_bytes) {
  w4_status st = check_dims(K, N, group, W4_F16);
  if (st) return st;
  if ((st = check_layout_dims(K, N, layout))) return st;
  const size_t G = (size_t)K / resolve_group(group, K);
  // TILE pads N to whole 128-column groups
  const size_t n_store = layout == W4_LAYOUT_TILE ? ((size_t)N + 127) / 128 * 128 : (size_t)N;
  if (qw_bytes) *qw_bytes = (size_t)K * n_store / 2;
  if (zeros_bytes) *zeros_bytes = G * N / 2;
  if (scales_bytes) *scales_bytes = G * N * 2;
  return W4_OK;
}

w4_status w4_repack_awq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int K,
                        int N, int group, int dtype, int layout, int32_t* qw_out,
                        int32_t* zeros_out, void* scales_out, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if ((st = check_layout_dims(K, N, layout))) return st;
  if (!qweight || !scales || !qw_out || !zeros_out || !scales_out) return W4_ERR_NULL;
  if (!aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) || !aligned16(qw_out) ||
      !aligned16(zeros_out) || !aligned16(scales_out))
    return W4_ERR_ALIGN;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  const size_t qw_b = (size_t)K * N / 2, z_b = G * N / 2, s_b = G * N * 2;
  size_t qw_out_b = 0;
  w4_repack_sizes(K, N, group, layout, &qw_out_b, nullptr, nullptr);
  const void* ins[3] = {qweight, qzeros, scales};
  const size_t in_b[3] = {qw_b, qzeros ? z_b : 0, s_b};
  const void* outs[3] = {qw_out, zeros_out, scales_out};
  const size_t out_b[3] = {qw_out_b, z_b, s_b};
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j)
      if (overlaps(outs[i], out_b[i], ins[j], in_b[j]) || (i != j && overlaps(outs[i], out_b[i], outs[j], out_b[j])))
        return W4_ERR_ALIAS;
  if ((st = check_arch())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = layout == W4_LAYOUT_STD ? launch_awq_to_std(qweight, qw_out, K, N, s)
                                          : launch_to_tile(qweight, 1, nullptr, qw_out, K, N, s);
  if (e != cudaSuccess) return W4_ERR_CUDA;
  if (launch_meta(qzeros, 1, scales, zeros_out, scales_out, (int)G, N, s) != cudaSuccess)
    return W4_ERR_CUDA;
  return from_cuda(launch_stream_fence(s));
}

w4_status w4_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                         const int32_t* g_idx, int K, int N, int group, int dtype, int layout,
                         int32_t* qw_out, int32_t* zeros_out, void* scales_out, int32_t* perm_out,
                         int32_t* status_out, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if ((st = check_layout_dims(K, N, layout))) return st;
  if (!qweight || !scales || !qw_out || !zeros_out || !scales_out) return W4_ERR_NULL;
  if (g_idx && (!perm_out || !status_out)) return W4_ERR_NULL;
  if (!aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) || !aligned16(qw_out) ||
      !aligned16(zeros_out) || !aligned16(scales_out) || !aligned16(g_idx) ||
      !aligned16(perm_out) || !aligned16(status_out))
    return W4_ERR_ALIGN;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  if (g_idx && G > (size_t)MAX_ACT_ORDER_GROUPS) return W4_ERR_SHAPE;
  const size_t qw_b = (size_t)K * N / 2, z_b = G * N / 2, s_b = G * N * 2;
  size_t qw_out_b = 0;
  w4_repack_sizes(K, N, group, layout, &qw_out_b, nullptr, nullptr);
  const size_t gi_b = g_idx ? (size_t)K * 4 : 0;
  const void* ins[4] = {qweight, qzeros, scales, g_idx};
  const size_t in_b[4] = {qw_b, qzeros ? z_b : 0, s_b, gi_b};
  const void* outs[5] = {qw_out, zeros_out, scales_out, g_idx ? perm_out : nullptr,
                         g_idx ? status_out : nullptr};
  const size_t out_b[5] = {qw_out_b, z_b, s_b, gi_b, g_idx ? (size_t)4 : 0};
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 4; ++j)
      if (overlaps(outs[i], out_b[i], ins[j], in_b[j])) return W4_ERR_ALIAS;
    for (int j = 0; j < 5; ++j)
      if (i != j && overlaps(outs[i], out_b[i], outs[j], out_b[j])) return W4_ERR_ALIAS;
  }
  if ((st = check_arch())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t* perm = nullptr;
  if (g_idx) {
    if (launch_act_order_perm(g_idx, K, g, perm_out, status_out, s) != cudaSuccess)
      return W4_ERR_CUDA;
    perm = perm_out;
  }
  cudaError_t e = layout == W4_LAYOUT_STD
                      ? launch_std_rows_permuted(qweight, perm, qw_out, K, N, s)
                      : launch_to_tile(qweight, 0, perm, qw_out, K, N, s);
  if (e != cudaSuccess) return W4_ERR_CUDA;
  if (launch_meta(qzeros, 0, scales, zeros_out, scales_out, (int)G, N, s) != cudaSuccess)
    return W4_ERR_CUDA;
  return from_cuda(launch_stream_fence(s));
}

size_t w4a16_gemm_workspace_size(int M, int N, int K, int group, int dtype, int has_perm) {
  (void)group;
  (void)dtype;
  // the small-M kernel: act-order calls stage x[:, perm] there once per call
  // (optional: without it every CTA gathers its own slice)
  if (M <= 16 || !prefill_supported(M, N, K)) return decode_workspace_bytes(M, K, has_perm != 0);
  // the tcgen05 kernel: the act-order staging is required, the split-K partials
  // after it are used when present
  const size_t staged = prefill_workspace_bytes(M, K, has_perm != 0);
  return staged + prefill_split_workspace_bytes(M, N, K);
}

w4_status w4_device_status(int32_t* status_out, int clear) {
  if (!status_out) return W4_ERR_NULL;
  int v = 0;
  if (read_device_status(&v, clear) != cudaSuccess) return W4_ERR_CUDA;
  *status_out = v;
  return W4_OK;
}

w4_status w4a16_gemm(const void* x, const int32_t* qw, const void* scales, const int32_t* zeros,
                     const int32_t* perm, void* y, int M, int N, int K, int group, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return w4a16_gemm_bias(x, qw, scales, zeros, perm, nullptr, y, M, N, K, group, dtype, workspace,
                         workspace_bytes, stream);
}

w4_status w4a16_gemm_bias(const void* x, const int32_t* qw, const void* scales,
                          const int32_t* zeros, const int32_t* perm, const void* bias, void* y,
                          int M, int N, int K, int group, int dtype, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return gemm_impl(x, qw, scales, zeros, perm, bias, y, M, N, K, group, dtype, workspace,
                   workspace_bytes, stream, 0);
}

w4_status w4a16_moe_gemm(const void* x, const int32_t* qw, const void* scales,
                         const int32_t* zeros, const int32_t* expert_offsets, void* y,
                         int num_experts, int max_rows_per_expert, int total_rows, int N, int K,
                         int group, int dtype, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if ((st = check_layout_dims(K, N, W4_LAYOUT_TILE))) return st;
  // more than 16 rows an expert: the tcgen05 kernel, when N is a multiple of
  // 32 (as w4a16_gemm routes M); otherwise the small-M kernel, up to 64 rows
  const bool large = max_rows_per_expert > 16 && grouped_prefill_supported(N, K, num_experts);
  if (num_experts < 1 || num_experts > 65535 || max_rows_per_expert < 1 ||
      max_rows_per_expert > (large ? MAX_DIM : DECODE_MAX_M) || total_rows < 0 ||
      total_rows > MAX_DIM)
    return W4_ERR_SHAPE;
  if (!qw || !scales || !zeros || !expert_offsets) return W4_ERR_NULL;
  if (total_rows > 0 && (!x || !y)) return W4_ERR_NULL;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(zeros) ||
      !aligned16(expert_offsets) || !aligned16(y))
    return W4_ERR_ALIGN;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  size_t qw_b = 0;
  w4_repack_sizes(K, N, group, W4_LAYOUT_TILE, &qw_b, nullptr, nullptr);
  const size_t E = (size_t)num_experts;
  const size_t y_b = (size_t)total_rows * N * 2;
  const void* ins[5] = {x, qw, scales, zeros, expert_offsets};
  const size_t in_b[5] = {(size_t)total_rows * K * 2, E * qw_b, E * G * N * 2, E * G * N / 2,
                          (E + 1) * 4};
  for (int j = 0; j < 5; ++j)
    if (overlaps(y, y_b, ins[j], in_b[j])) return W4_ERR_ALIAS;
  if ((st = check_arch())) return st;
  if (total_rows == 0) return W4_OK;
  GemmArgs a;
  a.x = x;
  a.qw = reinterpret_cast<const uint32_t*>(qw);
  a.scales = scales;
  a.zeros = reinterpret_cast<const uint32_t*>(zeros);
  a.perm = nullptr;
  a.y = y;
  a.bias = nullptr;
  a.M = max_rows_per_expert;
  a.N = N;
  a.K = K;
  a.group = g;
  a.bf16 = dtype == W4_BF16;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  a.eoff = expert_offsets;
  a.num_experts = num_experts;
  a.total_rows = total_rows;
  a.qw_estride = qw_b / 4;
  a.s_estride = G * N;
  a.z_estride = G * N / 8;
  if (large) return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
  return from_cuda(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

w4_status w4_test_stalled_gemm(const void* x, const int32_t* qw, const void* scales,
                               const int32_t* zeros, void* y, int M, int N, int K, int group,
                               int dtype, void* stream) {
  if (M < 1 || (M > 16 && !prefill_supported(M, N, K))) return W4_ERR_SHAPE;
  return gemm_impl(x, qw, scales, zeros, nullptr, nullptr, y, M, N, K, group, dtype, nullptr, 0,
                   stream, 1);
}

w4_status w4_test_prefill_plan(int M, int N, int K, int sm_count, int* out) {
  if (!out) return W4_ERR_NULL;
  if (M <= 16 || M > MAX_DIM || N < 1 || N > MAX_DIM || K < 1 || K > MAX_DIM || sm_count < 1 ||
      !prefill_supported(M, N, K))
    return W4_ERR_SHAPE;
  prefill_plan_query(M, N, K, sm_count, out);
  return W4_OK;
}

}  // extern "C"

namespace w4 {
namespace {

w4_status gemm_impl(const void* x, const int32_t* qw, const void* scales, const int32_t* zeros,
                    const int32_t* perm, const void* bias, void* y, int M, int N, int K,
                    int group, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                    int test_stall) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if (M < 0 || M > MAX_DIM) return W4_ERR_SHAPE;
  if ((st = check_layout_dims(K, N, W4_LAYOUT_TILE))) return st;
  if (!qw || !scales || !zeros) return W4_ERR_NULL;
  if (M > 0 && (!x || !y)) return W4_ERR_NULL;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(zeros) ||
      !aligned16(perm) || !aligned16(bias) || !aligned16(y) || !aligned16(workspace))
    return W4_ERR_ALIGN;
  // required: the act-order staging of the tcgen05 kernel (split-K partials are
  // optional and sized by the kernel from what the workspace holds)
  const size_t need = (M > 16 && prefill_supported(M, N, K))
                          ? prefill_workspace_bytes(M, K, perm != nullptr)
                          : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return W4_ERR_WORKSPACE;
  if (M == 0) return W4_OK;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  const size_t y_b = (size_t)M * N * 2;
  const void* ins[7] = {x, qw, scales, zeros, perm, workspace, bias};
  const size_t in_b[7] = {(size_t)M * K * 2, (size_t)K * N / 2, G * N * 2, G * N / 2,
                          perm ? (size_t)K * 4 : 0, workspace ? workspace_bytes : 0,
                          bias ? (size_t)N * 2 : 0};
  for (int j = 0; j < 7; ++j)
    if (overlaps(y, y_b, ins[j], in_b[j])) return W4_ERR_ALIAS;
  if ((st = check_arch())) return st;
  GemmArgs a;
  a.x = x;
  a.qw = reinterpret_cast<const uint32_t*>(qw);
  a.scales = scales;
  a.zeros = reinterpret_cast<const uint32_t*>(zeros);
  a.perm = perm;
  a.y = y;
  a.bias = bias;
  a.M = M;
  a.N = N;
  a.K = K;
  a.group = g;
  a.bf16 = dtype == W4_BF16;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.test_stall = test_stall;
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return W4_ERR_CUDA;
  if (use_prefill(M, N, K, info.sm_count))
    return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
  return from_cuda(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace w4

extern "C" {

w4_status w4a16_gemm_noalloc(const void* x, const int32_t* qw, const void* scales,
                             const int32_t* zeros, const int32_t* perm, void* y, int M, int N,
                             int K, int group, int dtype, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if (M < 0 || M > MAX_DIM) return W4_ERR_SHAPE;
  if ((st = check_layout_dims(K, N, W4_LAYOUT_TILE))) return st;
  const size_t need = (M > 16 && prefill_supported(M, N, K))
                          ? prefill_workspace_bytes(M, K, perm != nullptr)
                          : 0;
  if (need > W4_NOALLOC_SCRATCH_BYTES) return W4_ERR_WORKSPACE;
  // validate everything the scratch does not decide before touching the device
  st = w4a16_gemm(x, qw, scales, zeros, perm, y, 0, N, K, group, dtype, nullptr, 0, stream);
  if (st) return st;
  if (M == 0) return W4_OK;
  if (!x || !y) return W4_ERR_NULL;
  if ((st = check_arch())) return st;
  // the array's address is looked up on every path, so that the first call on
  // a device does the set-up whatever its shape
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (noalloc_scratch(&scratch, &scratch_bytes) != cudaSuccess) return W4_ERR_CUDA;
  if ((M <= 16 || !prefill_supported(M, N, K)) && perm == nullptr) {
    // the small-M kernel without act-order uses no workspace
    return w4a16_gemm(x, qw, scales, zeros, perm, y, M, N, K, group, dtype, nullptr, 0, stream);
  }
  return w4a16_gemm(x, qw, scales, zeros, perm, y, M, N, K, group, dtype, scratch, scratch_bytes,
                    stream);
}

size_t w4a8_gemm_workspace_size(int M, int K) {
  if (M < 1 || K < 1 || K > MAX_DIM || M > MAX_DIM || K % 128) return 0;
  return w4a8_workspace_bytes(M, K);
}

w4_status w4a8_gemm(const void* x, const int32_t* qw, const void* scales, const int32_t* zeros,
                    void* y, int M, int N, int K, int group, int dtype, void* workspace,
                    size_t workspace_bytes, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if (M < 0 || M > MAX_DIM) return W4_ERR_SHAPE;
  if ((st = check_layout_dims(K, N, W4_LAYOUT_TILE))) return st;
  if (group != 128 && group != -1) return W4_ERR_GROUP;
  if (K % 128 || N % 32) return W4_ERR_SHAPE;  // whole K blocks; zero rows of 16-byte multiples
  if (!qw || !scales || !zeros) return W4_ERR_NULL;
  if (M > 0 && (!x || !y || !workspace)) return W4_ERR_NULL;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(zeros) ||
      !aligned16(y) || !aligned16(workspace))
    return W4_ERR_ALIGN;
  if (M == 0) return W4_OK;
  if (workspace_bytes < w4a8_workspace_bytes(M, K)) return W4_ERR_WORKSPACE;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  const size_t y_b = (size_t)M * N * 2;
  size_t qw_b = 0;
  w4_repack_sizes(K, N, group, W4_LAYOUT_TILE, &qw_b, nullptr, nullptr);
  const void* ins[5] = {x, qw, scales, zeros, workspace};
  const size_t in_b[5] = {(size_t)M * K * 2, qw_b, G * N * 2, G * N / 2, workspace_bytes};
  for (int j = 0; j < 5; ++j)
    if (overlaps(y, y_b, ins[j], in_b[j])) return W4_ERR_ALIAS;
  if (overlaps(workspace, workspace_bytes, x, (size_t)M * K * 2)) return W4_ERR_ALIAS;
  if ((st = check_arch())) return st;
  return from_cuda(launch_w4a8(x, reinterpret_cast<const uint32_t*>(qw), scales,
                               reinterpret_cast<const uint32_t*>(zeros), y, M, N, K, g,
                               dtype == W4_BF16, workspace, static_cast<cudaStream_t>(stream)));
}

w4_status w4_dequant(const int32_t* qw, const void* scales, const int32_t* zeros, int K, int N,
                     int group, int dtype, int layout, int out_f32, void* w_out, void* stream) {
  w4_status st = check_dims(K, N, group, dtype);
  if (st) return st;
  if ((st = check_layout_dims(K, N, layout))) return st;
  if (!qw || !scales || !zeros || !w_out) return W4_ERR_NULL;
  if (!aligned16(qw) || !aligned16(scales) || !aligned16(zeros) || !aligned16(w_out))
    return W4_ERR_ALIGN;
  const int g = resolve_group(group, K);
  const size_t G = (size_t)K / g;
  const size_t w_b = (size_t)K * N * (out_f32 ? 4 : 2);
  if (overlaps(w_out, w_b, qw, (size_t)K * N / 2) || overlaps(w_out, w_b, scales, G * N * 2) ||
      overlaps(w_out, w_b, zeros, G * N / 2))
    return W4_ERR_ALIAS;
  if ((st = check_arch())) return st;
  return from_cuda(launch_dequant(qw, scales, zeros, K, N, g, dtype == W4_BF16, layout, out_f32,
                                  w_out, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
