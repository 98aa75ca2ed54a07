// gg_api.cu — the C ABI declared in include/gg.h: argument validation,
// workspace layout, device checks, and the composed forward / input-gradient
// of the expert layer. Host code only; kernels live in gg_permute.cu and
// gg_gemm.cu.
//
// Validation rules follow "perf(moe): add frozen grouped GEMM for adapter
// training" (AlignmentResearch/Megatron-LM PR #3), "Why existing behavior
// remains safe" (only grouped, frozen, bias-free BF16 expert weights; other
// configurations fail during preparation), NVIDIA/Megatron-LM PR #7333
// "Summary" (other GPU/library pairs fail explicitly) and "[Main] Support
// paged stash with device-initiated GroupedLinear" (NVIDIA/Megatron-LM PR
// #6828), "What does this PR do?" (reject instead of falling back).

#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "gg_internal.h"
#include "gg_mx.cuh"

namespace gg {

namespace {
std::atomic<uint64_t> g_launches{0};

struct DevCache {
  std::once_flag once;
  DeviceInfo info;
  gg_status status = GG_ERR_CUDA;
};
DevCache g_dev[kMaxDevices];

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline gg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GG_OK : GG_ERR_CUDA; }

inline int32_t* status_ptr(void* ws) { return static_cast<int32_t*>(ws); }

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

gg_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return GG_ERR_INVALID_ARG;
  if (!aligned16(ws)) return GG_ERR_MISALIGNED;
  if (ws_bytes < need) return GG_ERR_WORKSPACE_TOO_SMALL;
  return GG_OK;
}

gg_status device_ok(DeviceInfo* dev) {
  gg_status s = current_device(dev);
  if (s != GG_OK) return s;
  if (dev->cc_major != 10 || dev->cc_minor != 3) return GG_ERR_UNSUPPORTED_DEVICE;
  return GG_OK;
}

long long r_cap_of(int T, int k, int E, int P) {
  return static_cast<long long>(T) * k + static_cast<long long>(E) * (P - 1);
}
}  // namespace

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

gg_status current_device(DeviceInfo* out) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0) return GG_ERR_CUDA;
  if (d >= kMaxDevices) return GG_ERR_UNSUPPORTED_DEVICE;
  DevCache& c = g_dev[d];
  std::call_once(c.once, [&c, d] {
    DeviceInfo i;
    i.device = d;
    if (cudaDeviceGetAttribute(&i.sm_count, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&i.cc_major, cudaDevAttrComputeCapabilityMajor, d) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&i.cc_minor, cudaDevAttrComputeCapabilityMinor, d) !=
            cudaSuccess) {
      c.status = GG_ERR_CUDA;
      return;
    }
    c.info = i;
    c.status = GG_OK;
  });
  *out = c.info;
  return c.status;
}

}  // namespace gg

using namespace gg;

extern "C" {

const char* gg_status_string(int status) {
  switch (status) {
    case GG_OK: return "GG_OK";
    case GG_ERR_INVALID_ARG: return "GG_ERR_INVALID_ARG: invalid argument";
    case GG_ERR_UNSUPPORTED_SHAPE: return "GG_ERR_UNSUPPORTED_SHAPE: unsupported shape";
    case GG_ERR_MISALIGNED: return "GG_ERR_MISALIGNED: pointer not 16-byte aligned";
    case GG_ERR_WORKSPACE_TOO_SMALL: return "GG_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case GG_ERR_UNSUPPORTED_DEVICE:
      return "GG_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3";
    case GG_ERR_CUDA: return "GG_ERR_CUDA: a CUDA call failed";
    case GG_ERR_DEVICE_BAD_EXPERT_ID:
      return "GG_ERR_DEVICE_BAD_EXPERT_ID: expert id out of range";
    case GG_ERR_DEVICE_BAD_OFFSETS: return "GG_ERR_DEVICE_BAD_OFFSETS: invalid expert offsets";
    case GG_ERR_DEVICE_BAD_ROW: return "GG_ERR_DEVICE_BAD_ROW: row map entry out of range";
    case GG_ERR_DEVICE_TIMEOUT:
      return "GG_ERR_DEVICE_TIMEOUT: a bounded in-kernel wait ran out";
    default: return "unknown gg_status";
  }
}

const char* gg_version(void) { return "gg 0.2 sm_103a"; }

int gg_rowdot_blocks(int F) { return F > 0 ? 2 * ((F + 255) / 256) : 0; }

int gg_rowdot_stride(int F) { return (gg_rowdot_blocks(F) + 7) / 8 * 8; }

uint64_t gg_launch_count(void) { return g_launches.load(); }

size_t gg_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 0 || E <= 0) return 0;
  const long long R = static_cast<long long>(T) * k;
  const size_t hist = sizeof(int32_t) * static_cast<size_t>(permute_blocks(R)) * E;
  return kWsHeader + align256(hist);
}

gg_status gg_clear_status(void* ws, gg_stream_t stream) {
  if (ws == nullptr) return GG_ERR_INVALID_ARG;
  return from_cuda(
      cudaMemsetAsync(ws, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)));
}

gg_status gg_read_status(const void* ws, gg_stream_t stream, int32_t* host_status) {
  if (ws == nullptr || host_status == nullptr) return GG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return GG_ERR_CUDA;
  return from_cuda(cudaStreamSynchronize(s));
}

gg_status gg_permute(const gg_bf16* x, const int32_t* idx, const float* prob, int T, int H,
                     int k, int E, int pad_multiple, gg_bf16* Xp, int32_t* offsets,
                     int32_t* row_of_slot, int32_t* slot_of_row, float* prob_of_row, void* ws,
                     size_t ws_bytes, gg_stream_t stream) {
  if (T < 0 || H <= 0 || k <= 0 || E <= 0 || pad_multiple <= 0) return GG_ERR_INVALID_ARG;
  if (k > 32) return GG_ERR_INVALID_ARG;  // k > E is legal: duplicate ids share an expert
  if (E > kMaxExperts || H % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (r_cap_of(T, k, E, pad_multiple) > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  if (offsets == nullptr) return GG_ERR_INVALID_ARG;
  if (T > 0 && (idx == nullptr || prob == nullptr || row_of_slot == nullptr ||
                slot_of_row == nullptr || prob_of_row == nullptr))
    return GG_ERR_INVALID_ARG;
  if (T > 0 && Xp != nullptr && x == nullptr) return GG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Xp)) return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, gg_workspace_size(T, k, E));
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  int32_t* block_hist = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kWsHeader);
  return from_cuda(launch_permute(x, idx, prob, T, H, k, E, pad_multiple, Xp, offsets,
                                  row_of_slot, slot_of_row, prob_of_row, status_ptr(ws),
                                  block_hist, dev,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

gg_status gg_permute_rows(const gg_bf16* src, const int32_t* row_of_slot,
                          const int32_t* slot_of_row, const int32_t* offsets, int T, int H, int k,
                          int E, int pad_multiple, int R_cap, const float* prob, gg_bf16* dst,
                          void* ws, size_t ws_bytes, gg_stream_t stream) {
  if (T < 0 || H <= 0 || k <= 0 || k > 32 || E <= 0 || R_cap < 0 || pad_multiple <= 0)
    return GG_ERR_INVALID_ARG;
  if (E > kMaxExperts || H % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (offsets == nullptr || ws == nullptr) return GG_ERR_INVALID_ARG;
  if (R_cap > 0 && T > 0 &&
      (src == nullptr || row_of_slot == nullptr || slot_of_row == nullptr || dst == nullptr))
    return GG_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  return from_cuda(launch_gather_rows(src, row_of_slot, slot_of_row, offsets, H, k, E, R_cap, T,
                                      pad_multiple > 1, prob, dst, status_ptr(ws), dev.sm_count,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

static gg_status gemm_common_checks(const gg_bf16* A, const gg_bf16* B, const int32_t* offsets,
                                    int E, int R_cap, int K, int N, const gg_bf16* C, void* ws,
                                    size_t ws_bytes) {
  if (E <= 0 || R_cap < 0 || K <= 0 || N <= 0) return GG_ERR_INVALID_ARG;
  if (A == nullptr || B == nullptr || offsets == nullptr || C == nullptr)
    return GG_ERR_INVALID_ARG;
  if (E > kMaxExperts || K % 64 != 0 || N % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GG_ERR_MISALIGNED;
  return check_ws(ws, ws_bytes, kWsHeader);
}

static gg_status fwd_epilogue_checks(gg_epilogue epi, int N, const gg_bf16* H1_save,
                                     const float* prob_of_row) {
  const bool gated = epi == GG_EPI_SWIGLU || epi == GG_EPI_QGEGLU;
  if (epi != GG_EPI_NONE && !gated) return GG_ERR_INVALID_ARG;
  if (!gated && (H1_save != nullptr || prob_of_row != nullptr)) return GG_ERR_INVALID_ARG;
  if (gated && N % 128 != 0) return GG_ERR_UNSUPPORTED_SHAPE;  // F % 64
  if (!aligned16(H1_save)) return GG_ERR_MISALIGNED;
  return GG_OK;
}

gg_status gg_grouped_fwd(const gg_bf16* A, const gg_bf16* B, const int32_t* offsets, int E,
                         int R_cap, int K, int N, gg_epilogue epi, gg_bf16* C, gg_bf16* H1_save,
                         const float* prob_of_row, void* ws, size_t ws_bytes,
                         gg_stream_t stream) {
  gg_status s = gemm_common_checks(A, B, offsets, E, R_cap, K, N, C, ws, ws_bytes);
  if (s != GG_OK) return s;
  if ((s = fwd_epilogue_checks(epi, N, H1_save, prob_of_row)) != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  if (R_cap == 0) return GG_OK;
  GemmArgs a{};
  a.mode = epi == GG_EPI_NONE     ? kFwdPlain
           : epi == GG_EPI_QGEGLU ? kFwdQgeglu
                                  : kFwdSwiglu;
  a.row_scale = prob_of_row;
  a.A = A;
  a.B = B;
  a.offsets = offsets;
  a.E = E;
  a.R_cap = R_cap;
  a.Kred = K;
  a.Nout = N;
  a.Nw = N;
  a.Kw = K;
  a.C = C;
  a.H1_save = H1_save;
  a.status = status_ptr(ws);
  gg_status he = GG_OK;
  cudaError_t e = launch_grouped_gemm(a, dev, reinterpret_cast<cudaStream_t>(stream), &he);
  if (he != GG_OK) return he;
  return from_cuda(e);
}

gg_status gg_swiglu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap, int F,
                    gg_bf16* A, gg_stream_t stream) {
  return gg_glu(H1, offsets, E, R_cap, F, GG_EPI_SWIGLU, nullptr, A, stream);
}

gg_status gg_glu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap, int F,
                 gg_epilogue epi, const float* prob_of_row, gg_bf16* A, gg_stream_t stream) {
  if (E <= 0 || R_cap < 0 || F <= 0) return GG_ERR_INVALID_ARG;
  if (epi != GG_EPI_SWIGLU && epi != GG_EPI_QGEGLU) return GG_ERR_INVALID_ARG;
  if (H1 == nullptr || offsets == nullptr || A == nullptr) return GG_ERR_INVALID_ARG;
  if (E > kMaxExperts || F % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(H1) || !aligned16(A)) return GG_ERR_MISALIGNED;
  DeviceInfo dev;
  gg_status s = device_ok(&dev);
  if (s != GG_OK) return s;
  return from_cuda(launch_swiglu(H1, offsets, E, R_cap, F, glu_alpha(epi), prob_of_row, A,
                                 dev.sm_count,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

static gg_status dgrad_epilogue_checks(gg_epilogue epi, const gg_bf16* H1, const float* rowdot) {
  const bool gated = epi == GG_EPI_SWIGLU_BWD || epi == GG_EPI_QGEGLU_BWD;
  if (epi != GG_EPI_NONE && !gated) return GG_ERR_INVALID_ARG;
  if (!gated && (H1 != nullptr || rowdot != nullptr)) return GG_ERR_INVALID_ARG;
  if (gated && H1 == nullptr) return GG_ERR_INVALID_ARG;
  if (!aligned16(H1) || (reinterpret_cast<uintptr_t>(rowdot) & 31u) != 0) return GG_ERR_MISALIGNED;
  return GG_OK;
}

gg_status gg_grouped_dgrad(const gg_bf16* dC, const gg_bf16* B, const int32_t* offsets, int E,
                           int R_cap, int K, int N, gg_epilogue epi, const gg_bf16* H1,
                           const float* prob_of_row, gg_bf16* dA, float* rowdot, void* ws,
                           size_t ws_bytes, gg_stream_t stream) {
  gg_status s = gemm_common_checks(dC, B, offsets, E, R_cap, K, N, dA, ws, ws_bytes);
  if (s != GG_OK) return s;
  if ((s = dgrad_epilogue_checks(epi, H1, rowdot)) != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  if (R_cap == 0) return GG_OK;
  GemmArgs a{};
  a.mode = epi == GG_EPI_NONE         ? kDgradPlain
           : epi == GG_EPI_QGEGLU_BWD ? kDgradQgegluBwd
                                      : kDgradSwigluBwd;
  a.A = dC;
  a.B = B;
  a.offsets = offsets;
  a.E = E;
  a.R_cap = R_cap;
  a.Kred = N;
  a.Nout = K;
  a.Nw = N;
  a.Kw = K;
  a.C = dA;
  a.H1 = H1;
  a.row_scale = prob_of_row;
  a.rowdot = rowdot;
  a.status = status_ptr(ws);
  gg_status he = GG_OK;
  cudaError_t e = launch_grouped_gemm(a, dev, reinterpret_cast<cudaStream_t>(stream), &he);
  if (he != GG_OK) return he;
  return from_cuda(e);
}

static gg_status gather_checks(const gg_bf16* src, int T, const int32_t* slot_of_row, int k) {
  if (T < 0 || k <= 0 || src == nullptr || slot_of_row == nullptr) return GG_ERR_INVALID_ARG;
  if (!aligned16(src)) return GG_ERR_MISALIGNED;
  return GG_OK;
}

gg_status gg_grouped_fwd_gather(const gg_bf16* src, int T, const int32_t* slot_of_row, int k,
                                const gg_bf16* B, const int32_t* offsets, int E, int R_cap, int K,
                                int N, gg_epilogue epi, gg_bf16* C, gg_bf16* H1_save,
                                const float* prob_of_row, void* ws, size_t ws_bytes,
                                gg_stream_t stream) {
  gg_status s = gather_checks(src, T, slot_of_row, k);
  if (s != GG_OK) return s;
  // the source stands in for A in the common checks
  s = gemm_common_checks(src, B, offsets, E, R_cap, K, N, C, ws, ws_bytes);
  if (s != GG_OK) return s;
  if ((s = fwd_epilogue_checks(epi, N, H1_save, prob_of_row)) != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  if (R_cap == 0 || T == 0) return GG_OK;
  GemmArgs a{};
  a.mode = epi == GG_EPI_NONE     ? kFwdPlain
           : epi == GG_EPI_QGEGLU ? kFwdQgeglu
                                  : kFwdSwiglu;
  a.row_scale = prob_of_row;
  a.B = B;
  a.offsets = offsets;
  a.E = E;
  a.R_cap = R_cap;
  a.Kred = K;
  a.Nout = N;
  a.Nw = N;
  a.Kw = K;
  a.C = C;
  a.H1_save = H1_save;
  a.status = status_ptr(ws);
  a.gather_src = src;
  a.slot_of_row = slot_of_row;
  a.gather_k = k;
  a.gather_rows = T;
  gg_status he = GG_OK;
  cudaError_t e = launch_grouped_gemm(a, dev, reinterpret_cast<cudaStream_t>(stream), &he);
  if (he != GG_OK) return he;
  return from_cuda(e);
}

gg_status gg_grouped_dgrad_gather(const gg_bf16* src, int T, const int32_t* slot_of_row, int k,
                                  const gg_bf16* B, const int32_t* offsets, int E, int R_cap,
                                  int K, int N, gg_epilogue epi, const gg_bf16* H1,
                                  const float* prob_of_row, gg_bf16* dA, float* rowdot, void* ws,
                                  size_t ws_bytes, gg_stream_t stream) {
  gg_status s = gather_checks(src, T, slot_of_row, k);
  if (s != GG_OK) return s;
  s = gemm_common_checks(src, B, offsets, E, R_cap, K, N, dA, ws, ws_bytes);
  if (s != GG_OK) return s;
  if ((s = dgrad_epilogue_checks(epi, H1, rowdot)) != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  if (R_cap == 0 || T == 0) return GG_OK;
  GemmArgs a{};
  a.mode = epi == GG_EPI_NONE         ? kDgradPlain
           : epi == GG_EPI_QGEGLU_BWD ? kDgradQgegluBwd
                                      : kDgradSwigluBwd;
  a.B = B;
  a.offsets = offsets;
  a.E = E;
  a.R_cap = R_cap;
  a.Kred = N;
  a.Nout = K;
  a.Nw = N;
  a.Kw = K;
  a.C = dA;
  a.H1 = H1;
  a.row_scale = prob_of_row;
  a.rowdot = rowdot;
  a.status = status_ptr(ws);
  a.gather_src = src;
  a.slot_of_row = slot_of_row;
  a.gather_k = k;
  a.gather_rows = T;
  gg_status he = GG_OK;
  cudaError_t e = launch_grouped_gemm(a, dev, reinterpret_cast<cudaStream_t>(stream), &he);
  if (he != GG_OK) return he;
  return from_cuda(e);
}

gg_status gg_unpermute_combine(const gg_bf16* Yp, const int32_t* row_of_slot, const float* prob,
                               int T, int k, int H, int R_cap, gg_bf16* out, const float* rowdot,
                               int n_rowdot, const gg_bf16* dot_src, float* dprob, void* ws,
                               size_t ws_bytes, gg_stream_t stream) {
  if (T < 0 || k <= 0 || k > 32 || H <= 0 || R_cap < 0) return GG_ERR_INVALID_ARG;
  if (H % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (Yp == nullptr || row_of_slot == nullptr || out == nullptr))
    return GG_ERR_INVALID_ARG;
  // dprob needs exactly one source: the partial sums or the token-major rows
  if (dprob != nullptr && (rowdot != nullptr) == (dot_src != nullptr)) return GG_ERR_INVALID_ARG;
  if (dprob != nullptr && rowdot != nullptr && n_rowdot <= 0) return GG_ERR_INVALID_ARG;
  if (dprob == nullptr && (rowdot != nullptr || dot_src != nullptr)) return GG_ERR_INVALID_ARG;
  if (!aligned16(dot_src)) return GG_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(rowdot) & 31u) != 0) return GG_ERR_MISALIGNED;
  if (!aligned16(Yp) || !aligned16(out)) return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  return from_cuda(launch_combine(Yp, row_of_slot, prob, T, k, H, R_cap, out, rowdot,
                                  rowdot != nullptr ? n_rowdot : 0, dot_src, nullptr, dprob,
                                  status_ptr(ws), dev.sm_count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

gg_status gg_unpermute_combine_dot(const gg_bf16* Sp, const int32_t* row_of_slot,
                                   const float* prob, int T, int k, int H, int R_cap,
                                   gg_bf16* out, const gg_bf16* dot_src, const gg_bf16* dot_rows,
                                   float* dprob, void* ws, size_t ws_bytes, gg_stream_t stream) {
  if (T < 0 || k <= 0 || k > 32 || H <= 0 || R_cap < 0) return GG_ERR_INVALID_ARG;
  if (H % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (Sp == nullptr || row_of_slot == nullptr || out == nullptr ||
                dot_src == nullptr || dot_rows == nullptr || dprob == nullptr))
    return GG_ERR_INVALID_ARG;
  if (!aligned16(Sp) || !aligned16(out) || !aligned16(dot_src) || !aligned16(dot_rows))
    return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  return from_cuda(launch_combine(Sp, row_of_slot, prob, T, k, H, R_cap, out, nullptr, 0,
                                  dot_src, dot_rows, dprob, status_ptr(ws), dev.sm_count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------ expert parallelism

gg_status gg_ep_split_ids(const int32_t* idx, int n, int El, int n_ranks, int32_t* dest,
                          int32_t* local_eid, void* ws, size_t ws_bytes, gg_stream_t stream) {
  if (n < 0 || El <= 0 || n_ranks <= 0) return GG_ERR_INVALID_ARG;
  if (static_cast<long long>(El) * n_ranks > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  if (n > 0 && (idx == nullptr || dest == nullptr || local_eid == nullptr))
    return GG_ERR_INVALID_ARG;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  return from_cuda(launch_ep_split_ids(idx, n, El, n_ranks, dest, local_eid, status_ptr(ws),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

gg_status gg_gather_rows32(const void* src, int src_rows, int width, const int32_t* index,
                           int n, void* out, void* ws, size_t ws_bytes, gg_stream_t stream) {
  if (n < 0 || src_rows < 0 || width <= 0) return GG_ERR_INVALID_ARG;
  if (n > 0 && (src == nullptr && src_rows > 0)) return GG_ERR_INVALID_ARG;
  if (n > 0 && (index == nullptr || out == nullptr)) return GG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  return from_cuda(launch_gather_rows32(static_cast<const uint32_t*>(src), src_rows, width, index,
                                        n, static_cast<uint32_t*>(out), status_ptr(ws),
                                        dev.sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ composite

size_t gg_moe_buffers_size(int T, int H, int F, int k, int E, int pad_multiple) {
  if (T < 0 || H <= 0 || F <= 0 || k <= 0 || E <= 0 || pad_multiple <= 0) return 0;
  const size_t R_cap = static_cast<size_t>(r_cap_of(T, k, E, pad_multiple));
  const size_t b2 = sizeof(gg_bf16);
  size_t n = 0;
  n += align256(R_cap * H * b2) * 4;         // Xp, Yp, dYp, dXp
  n += align256(R_cap * 2 * F * b2) * 2;     // H1, dH
  n += align256(R_cap * F * b2);             // A
  n += align256(sizeof(int32_t) * (E + 1));  // offsets
  n += align256(sizeof(int32_t) * static_cast<size_t>(T) * k);  // row_of_slot
  n += align256(sizeof(int32_t) * R_cap);    // slot_of_row
  n += align256(sizeof(float) * R_cap);      // prob_of_row
  n += align256(sizeof(float) * R_cap * gg_rowdot_stride(F));  // rowdot
  n += align256(gg_workspace_size(T, k, E)); // workspace (status first)
  return n;
}

gg_status gg_moe_buffers_bind(void* base, size_t bytes, int T, int H, int F, int k, int E,
                              int pad_multiple, gg_moe_buffers* out) {
  if (base == nullptr || out == nullptr) return GG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(base) & 255u) return GG_ERR_MISALIGNED;
  const size_t need = gg_moe_buffers_size(T, H, F, k, E, pad_multiple);
  if (need == 0) return GG_ERR_INVALID_ARG;
  if (bytes < need) return GG_ERR_WORKSPACE_TOO_SMALL;
  const size_t R_cap = static_cast<size_t>(r_cap_of(T, k, E, pad_multiple));
  uint8_t* p = static_cast<uint8_t*>(base);
  auto take = [&p](size_t n) {
    uint8_t* q = p;
    p += align256(n);
    return q;
  };
  const size_t b2 = sizeof(gg_bf16);
  std::memset(out, 0, sizeof(*out));
  out->Xp = reinterpret_cast<gg_bf16*>(take(R_cap * H * b2));
  out->Yp = reinterpret_cast<gg_bf16*>(take(R_cap * H * b2));
  out->dYp = reinterpret_cast<gg_bf16*>(take(R_cap * H * b2));
  out->dXp = reinterpret_cast<gg_bf16*>(take(R_cap * H * b2));
  out->H1 = reinterpret_cast<gg_bf16*>(take(R_cap * 2 * F * b2));
  out->dH = reinterpret_cast<gg_bf16*>(take(R_cap * 2 * F * b2));
  out->A = reinterpret_cast<gg_bf16*>(take(R_cap * F * b2));
  out->offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  out->row_of_slot =
      reinterpret_cast<int32_t*>(take(sizeof(int32_t) * static_cast<size_t>(T) * k));
  out->slot_of_row = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * R_cap));
  out->prob_of_row = reinterpret_cast<float*>(take(sizeof(float) * R_cap));
  out->rowdot = reinterpret_cast<float*>(take(sizeof(float) * R_cap * gg_rowdot_stride(F)));
  out->ws_bytes = align256(gg_workspace_size(T, k, E));
  out->ws = take(out->ws_bytes);
  return GG_OK;
}

static gg_status check_buffers(const gg_moe_buffers* b, int T, int k, int E) {
  if (b == nullptr) return GG_ERR_INVALID_ARG;
  if (b->Xp == nullptr || b->H1 == nullptr || b->A == nullptr || b->Yp == nullptr ||
      b->dYp == nullptr || b->dH == nullptr || b->dXp == nullptr || b->offsets == nullptr ||
      b->row_of_slot == nullptr || b->slot_of_row == nullptr || b->prob_of_row == nullptr ||
      b->rowdot == nullptr)
    return GG_ERR_INVALID_ARG;
  return check_ws(b->ws, b->ws_bytes, gg_workspace_size(T, k, E));
}

static gg_status read_options(const gg_moe_options* opt, gg_epilogue* fwd_epi,
                              gg_epilogue* bwd_epi, int* mode, bool* recompute) {
  const int act = opt != nullptr ? opt->activation : GG_ACT_SWIGLU;
  *mode = opt != nullptr ? opt->prob_mode : GG_PROB_COMBINE;
  *recompute = opt != nullptr && opt->recompute_h1 != 0;
  if (opt != nullptr && opt->recompute_h1 != 0 && opt->recompute_h1 != 1)
    return GG_ERR_INVALID_ARG;
  if (act != GG_ACT_SWIGLU && act != GG_ACT_QGEGLU) return GG_ERR_INVALID_ARG;
  if (*mode != GG_PROB_COMBINE && *mode != GG_PROB_ACTIVATION && *mode != GG_PROB_PRE_FC1)
    return GG_ERR_INVALID_ARG;
  *fwd_epi = act == GG_ACT_QGEGLU ? GG_EPI_QGEGLU : GG_EPI_SWIGLU;
  *bwd_epi = act == GG_ACT_QGEGLU ? GG_EPI_QGEGLU_BWD : GG_EPI_SWIGLU_BWD;
  return GG_OK;
}

gg_status gg_moe_mlp_fwd_ex(const gg_bf16* x, const int32_t* idx, const float* prob,
                            const gg_bf16* W1, const gg_bf16* W2, int T, int H, int F, int k,
                            int E, int pad_multiple, const gg_moe_options* opt, gg_bf16* out,
                            const gg_moe_buffers* buf, gg_stream_t stream) {
  if (T < 0 || H <= 0 || k <= 0 || E <= 0 || pad_multiple <= 0) return GG_ERR_INVALID_ARG;
  gg_epilogue fepi, bepi;
  int mode;
  bool recompute;
  gg_status s = read_options(opt, &fepi, &bepi, &mode, &recompute);
  if (s != GG_OK) return s;
  if ((s = check_buffers(buf, T, k, E)) != GG_OK) return s;
  if (W1 == nullptr || W2 == nullptr || F <= 0) return GG_ERR_INVALID_ARG;
  if (F % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && out == nullptr) return GG_ERR_INVALID_ARG;
  const long long rc = r_cap_of(T, k, E, pad_multiple);
  if (rc > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  const int R_cap = static_cast<int>(rc);
  if (T > 0 && x == nullptr) return GG_ERR_INVALID_ARG;
  // The permuted copy of x is written once by a bandwidth-bound row copy and
  // read by FC1's tile loads: on GB300 this is several times cheaper than
  // four-row TMA gathers inside FC1 (gg_grouped_fwd_gather), which re-gather
  // every A row once per column block. Before FC1 the copy takes the
  // probability along (GG_PROB_PRE_FC1).
  const bool pre = mode == GG_PROB_PRE_FC1;
  s = gg_permute(x, idx, prob, T, H, k, E, pad_multiple, pre ? nullptr : buf->Xp, buf->offsets,
                 buf->row_of_slot, buf->slot_of_row, buf->prob_of_row, buf->ws, buf->ws_bytes,
                 stream);
  if (s != GG_OK || T == 0) return s;
  if (pre) {
    s = gg_permute_rows(x, buf->row_of_slot, buf->slot_of_row, buf->offsets, T, H, k, E,
                        pad_multiple, R_cap, prob, buf->Xp, buf->ws, buf->ws_bytes, stream);
    if (s != GG_OK) return s;
  }
  s = gg_grouped_fwd(buf->Xp, W1, buf->offsets, E, R_cap, H, 2 * F, fepi, buf->A,
                     recompute ? nullptr : buf->H1,
                     mode == GG_PROB_ACTIVATION ? buf->prob_of_row : nullptr, buf->ws,
                     buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  s = gg_grouped_fwd(buf->A, W2, buf->offsets, E, R_cap, F, H, GG_EPI_NONE, buf->Yp, nullptr,
                     nullptr, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  return gg_unpermute_combine(buf->Yp, buf->row_of_slot, mode == GG_PROB_COMBINE ? prob : nullptr,
                              T, k, H, R_cap, out, nullptr, 0, nullptr, nullptr, buf->ws,
                              buf->ws_bytes, stream);
}

gg_status gg_moe_mlp_fwd(const gg_bf16* x, const int32_t* idx, const float* prob,
                         const gg_bf16* W1, const gg_bf16* W2, int T, int H, int F, int k, int E,
                         int pad_multiple, gg_bf16* out, const gg_moe_buffers* buf,
                         gg_stream_t stream) {
  return gg_moe_mlp_fwd_ex(x, idx, prob, W1, W2, T, H, F, k, E, pad_multiple, nullptr, out, buf,
                           stream);
}

gg_status gg_moe_mlp_bwd_ex(const gg_bf16* dOut, const gg_bf16* x, const float* prob,
                            const gg_bf16* W1, const gg_bf16* W2, int T, int H, int F, int k,
                            int E, int pad_multiple, const gg_moe_options* opt, gg_bf16* dX,
                            float* dprob, const gg_moe_buffers* buf, gg_stream_t stream) {
  if (T < 0 || H <= 0 || k <= 0 || E <= 0 || pad_multiple <= 0 || F <= 0)
    return GG_ERR_INVALID_ARG;
  gg_epilogue fepi, bepi;
  int mode;
  bool recompute;
  gg_status s = read_options(opt, &fepi, &bepi, &mode, &recompute);
  if (s != GG_OK) return s;
  if ((s = check_buffers(buf, T, k, E)) != GG_OK) return s;
  if (W1 == nullptr || W2 == nullptr) return GG_ERR_INVALID_ARG;
  if (F % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return GG_OK;
  if (dOut == nullptr || dX == nullptr) return GG_ERR_INVALID_ARG;
  const bool pre = mode == GG_PROB_PRE_FC1;
  if (pre && (prob == nullptr || (dprob != nullptr && x == nullptr))) return GG_ERR_INVALID_ARG;
  const long long rc = r_cap_of(T, k, E, pad_multiple);
  if (rc > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  const int R_cap = static_cast<int>(rc);
  float* rowdot = dprob != nullptr && !pre ? buf->rowdot : nullptr;
  if (recompute) {  // H1 = bf16(Xp_e @ W1_e^T), the bits the forward's epilogue would store
    s = gg_grouped_fwd(buf->Xp, W1, buf->offsets, E, R_cap, H, 2 * F, GG_EPI_NONE, buf->H1,
                       nullptr, nullptr, buf->ws, buf->ws_bytes, stream);
    if (s != GG_OK) return s;
  }
  s = gg_permute_rows(dOut, buf->row_of_slot, buf->slot_of_row, buf->offsets, T, H, k, E,
                      pad_multiple, R_cap, nullptr, buf->dYp, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  // dH = act'(H1) applied to [prob_of_row *] (dYp @ W2_e), W2 being [E][H][F]:
  // the probability scales the activation's gradient unless it was applied
  // before FC1
  s = gg_grouped_dgrad(buf->dYp, W2, buf->offsets, E, R_cap, F, H, bepi, buf->H1,
                       pre ? nullptr : buf->prob_of_row, buf->dH, rowdot, buf->ws,
                       buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  // dXp = dH @ W1_e; W1 is [E][2F][H]
  s = gg_grouped_dgrad(buf->dH, W1, buf->offsets, E, R_cap, H, 2 * F, GG_EPI_NONE, nullptr,
                       nullptr, buf->dXp, nullptr, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  if (pre)  // Xp = prob * x: dX = sum_j prob * dXp[row], dprob = <x_t, dXp[row]>
    return gg_unpermute_combine(buf->dXp, buf->row_of_slot, prob, T, k, H, R_cap, dX, nullptr, 0,
                                dprob != nullptr ? x : nullptr, dprob, buf->ws, buf->ws_bytes,
                                stream);
  return gg_unpermute_combine(buf->dXp, buf->row_of_slot, nullptr, T, k, H, R_cap, dX, rowdot,
                              gg_rowdot_blocks(F), nullptr, dprob, buf->ws, buf->ws_bytes,
                              stream);
}

gg_status gg_moe_mlp_bwd(const gg_bf16* dOut, const gg_bf16* W1, const gg_bf16* W2, int T, int H,
                         int F, int k, int E, int pad_multiple, gg_bf16* dX, float* dprob,
                         const gg_moe_buffers* buf, gg_stream_t stream) {
  return gg_moe_mlp_bwd_ex(dOut, nullptr, nullptr, W1, W2, T, H, F, k, E, pad_multiple, nullptr,
                           dX, dprob, buf, stream);
}

// ------------------------------------------------------------------ MXFP8

static bool mx_shape_ok(int E, int H, int F) {
  return E > 0 && E <= kMaxExperts && H > 0 && F > 0 && H % 128 == 0 && F % 128 == 0;
}

int gg_mx_row_tiles(int T, int k, int E, int pad_multiple) {
  if (T < 0 || k <= 0 || E <= 0 || pad_multiple <= 0) return 0;
  const long long rc = r_cap_of(T, k, E, pad_multiple);
  const long long n = (rc + 127) / 128 + E;
  return n > 0x7FFFFFFFLL ? 0 : static_cast<int>(n);
}

// the SwiGLU-backward GEMM runs 128-column tiles: two partials per tile
int gg_mx_rowdot_blocks(int F) { return F > 0 ? 2 * ((F + 127) / 128) : 0; }

int gg_mx_rowdot_stride(int F) { return (gg_mx_rowdot_blocks(F) + 7) / 8 * 8; }

gg_status gg_mx_weights_layout_of(int E, int H, int F, gg_mx_weights_layout* out) {
  if (out == nullptr) return GG_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, H, F)) return GG_ERR_UNSUPPORTED_SHAPE;
  const size_t e = static_cast<size_t>(E), h = static_cast<size_t>(H), f = static_cast<size_t>(F);
  const size_t sfb = mx::kSfbBytes;
  const size_t tn = mx::kTileN, th = mx::kTileNHalf;
  size_t at = 0;
  auto take = [&at](size_t n) {
    const size_t q = at;
    at += align256(n);
    return q;
  };
  out->w1 = take(e * 2 * f * h);
  out->w1_scales = take(e * ((f + th - 1) / th) * (h / 128) * sfb);
  out->w2 = take(e * h * f);
  out->w2_scales = take(e * ((h + tn - 1) / tn) * (f / 128) * sfb);
  out->w2t = take(e * f * h);
  out->w2t_scales = take(e * ((f + tn - 1) / tn) * (h / 128) * sfb);
  out->w1t = take(e * h * 2 * f);
  out->w1t_scales = take(e * ((h + tn - 1) / tn) * (2 * f / 128) * sfb);
  out->bytes = at;
  return GG_OK;
}

gg_status gg_mx_prepare_weights(const gg_bf16* W1, const gg_bf16* W2, int E, int H, int F,
                                void* mxw, size_t bytes, gg_stream_t stream) {
  gg_mx_weights_layout L;
  gg_status s = gg_mx_weights_layout_of(E, H, F, &L);
  if (s != GG_OK) return s;
  if (W1 == nullptr || W2 == nullptr || mxw == nullptr) return GG_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || (reinterpret_cast<uintptr_t>(mxw) & 255u) != 0)
    return GG_ERR_MISALIGNED;
  if (bytes < L.bytes) return GG_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(mxw);
  // scale bytes of columns past a weight's rows stay 0
  const size_t scale_regions[4][2] = {{L.w1_scales, L.w2 - L.w1_scales},
                                      {L.w2_scales, L.w2t - L.w2_scales},
                                      {L.w2t_scales, L.w1t - L.w2t_scales},
                                      {L.w1t_scales, L.bytes - L.w1t_scales}};
  for (const auto& r : scale_regions) {
    cudaError_t e = cudaMemsetAsync(base + r[0], 0, r[1], st);
    if (e != cudaSuccess) return GG_ERR_CUDA;
  }
  const int tn = mx::kTileN, th = mx::kTileNHalf;
  if (launch_mx_prepare_weight(W1, E, 2 * F, H, false, F, (F + th - 1) / th, base + L.w1,
                               base + L.w1_scales, st) != cudaSuccess ||
      launch_mx_prepare_weight(W2, E, H, F, false, 0, (H + tn - 1) / tn, base + L.w2,
                               base + L.w2_scales, st) != cudaSuccess ||
      launch_mx_prepare_weight(W2, E, F, H, true, 0, (F + tn - 1) / tn, base + L.w2t,
                               base + L.w2t_scales, st) != cudaSuccess ||
      launch_mx_prepare_weight(W1, E, H, 2 * F, true, 0, (H + tn - 1) / tn, base + L.w1t,
                               base + L.w1t_scales, st) != cudaSuccess)
    return GG_ERR_CUDA;
  return GG_OK;
}

gg_status gg_mx_quantize_rows(const gg_bf16* src, int T, int K, int k,
                              const int32_t* row_of_slot, const int32_t* slot_of_row,
                              const int32_t* offsets, const float* prob, int E,
                              int pad_multiple, int n_tiles, int32_t* tiles_before, uint8_t* Q,
                              uint8_t* S, void* ws, size_t ws_bytes, gg_stream_t stream) {
  if (T < 0 || K <= 0 || k <= 0 || k > 32 || E <= 0 || pad_multiple <= 0 || n_tiles < 0)
    return GG_ERR_INVALID_ARG;
  if (E > kMaxExperts || K % 128 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  const long long rc = r_cap_of(T, k, E, pad_multiple);
  if (rc > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  const int R_cap = static_cast<int>(rc);
  if (offsets == nullptr || tiles_before == nullptr || S == nullptr) return GG_ERR_INVALID_ARG;
  if (T > 0 && (src == nullptr || row_of_slot == nullptr || slot_of_row == nullptr ||
                Q == nullptr))
    return GG_ERR_INVALID_ARG;
  if (n_tiles < (R_cap + 127) / 128 + E) return GG_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(src) || !aligned16(Q) || !aligned16(S)) return GG_ERR_MISALIGNED;
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_mx_tile_prefix(offsets, E, tiles_before, st);
  if (e != cudaSuccess) return GG_ERR_CUDA;
  return from_cuda(launch_mx_quantize_rows(src, T, K, k, row_of_slot, slot_of_row, offsets,
                                           tiles_before, E, R_cap, pad_multiple > 1, n_tiles,
                                           prob, Q, S, status_ptr(ws), dev.sm_count, st));
}

gg_status gg_mx_grouped_gemm(int which, int activation, const uint8_t* Aq, const uint8_t* As,
                             const void* mxw, const int32_t* offsets, int E, int R_cap, int H,
                             int F, int n_tiles, gg_bf16* C, uint8_t* Cq, uint8_t* Cs,
                             gg_bf16* H1, const float* row_scale, float* rowdot, void* ws,
                             size_t ws_bytes, gg_stream_t stream) {
  if (R_cap < 0 || n_tiles < 0) return GG_ERR_INVALID_ARG;
  if (activation != GG_ACT_SWIGLU && activation != GG_ACT_QGEGLU) return GG_ERR_INVALID_ARG;
  gg_mx_weights_layout L;
  gg_status s = gg_mx_weights_layout_of(E, H, F, &L);
  if (s != GG_OK) return s;
  if (n_tiles < (R_cap + 127) / 128 + E) return GG_ERR_WORKSPACE_TOO_SMALL;
  if (Aq == nullptr || As == nullptr || mxw == nullptr || offsets == nullptr)
    return GG_ERR_INVALID_ARG;
  const bool qg = activation == GG_ACT_QGEGLU;
  const uint8_t* w = static_cast<const uint8_t*>(mxw);
  MxGemmArgs a{};
  a.A = Aq;
  a.As = As;
  a.sf_tiles = n_tiles;
  a.offsets = offsets;
  a.E = E;
  a.R_cap = R_cap;
  a.C = C;
  a.Cq = Cq;
  a.Cs = Cs;
  a.row_scale = row_scale;
  switch (which) {
    case GG_MX_FC1:
      if (Cq == nullptr || Cs == nullptr || rowdot != nullptr) return GG_ERR_INVALID_ARG;
      a.mode = qg ? kFwdQgeglu : kFwdSwiglu;
      a.K = H, a.Nout = 2 * F, a.Nw = 2 * F, a.Kq = F;
      a.B = w + L.w1, a.Bs = w + L.w1_scales;
      a.H1_save = H1;
      break;
    case GG_MX_FC2:
      if (C == nullptr || row_scale != nullptr || rowdot != nullptr) return GG_ERR_INVALID_ARG;
      a.mode = kFwdPlain;
      a.K = F, a.Nout = H, a.Nw = H;
      a.B = w + L.w2, a.Bs = w + L.w2_scales;
      break;
    case GG_MX_DGRAD_FC2:
      if (Cq == nullptr || Cs == nullptr || H1 == nullptr) return GG_ERR_INVALID_ARG;
      a.mode = qg ? kDgradQgegluBwd : kDgradSwigluBwd;
      a.K = H, a.Nout = F, a.Nw = F, a.Kq = 2 * F;
      a.B = w + L.w2t, a.Bs = w + L.w2t_scales;
      a.H1 = H1;
      a.rowdot = rowdot;
      break;
    case GG_MX_DGRAD_FC1:
      if (C == nullptr || rowdot != nullptr) return GG_ERR_INVALID_ARG;
      a.mode = kDgradPlain;
      a.K = 2 * F, a.Nout = H, a.Nw = H;
      a.B = w + L.w1t, a.Bs = w + L.w1t_scales;
      break;
    default:
      return GG_ERR_INVALID_ARG;
  }
  if (!aligned16(Aq) || !aligned16(As) || !aligned16(C) || !aligned16(Cq) || !aligned16(H1) ||
      (reinterpret_cast<uintptr_t>(mxw) & 255u) != 0)
    return GG_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(rowdot) & 31u) != 0) return GG_ERR_MISALIGNED;
  if ((s = check_ws(ws, ws_bytes, kWsHeader)) != GG_OK) return s;
  if (R_cap == 0) return GG_OK;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  a.status = status_ptr(ws);
  gg_status he = GG_OK;
  const cudaError_t e =
      launch_grouped_gemm_mx(a, dev, reinterpret_cast<cudaStream_t>(stream), &he);
  if (he != GG_OK) return he;
  return from_cuda(e);
}

size_t gg_mx_buffers_size(int T, int H, int F, int k, int E, int pad_multiple) {
  if (T < 0 || k <= 0 || pad_multiple <= 0 || !mx_shape_ok(E, H, F)) return 0;
  const size_t R_cap = static_cast<size_t>(r_cap_of(T, k, E, pad_multiple));
  const size_t nt = static_cast<size_t>(gg_mx_row_tiles(T, k, E, pad_multiple));
  const size_t h = static_cast<size_t>(H), f = static_cast<size_t>(F);
  size_t n = 0;
  n += align256(R_cap * h) * 2 + align256(nt * (h / 128) * 512) * 2;   // Xq, dYq + scales
  n += align256(R_cap * f) + align256(nt * (f / 128) * 512);            // Aq + scales
  n += align256(R_cap * 2 * f) + align256(nt * (2 * f / 128) * 512);    // dHq + scales
  n += align256(R_cap * 2 * f * 2);                                     // H1
  n += align256(R_cap * h * 2) * 2;                                     // Yp, dXp
  n += align256(sizeof(int32_t) * (E + 1)) * 2;                         // offsets, tiles_before
  n += align256(sizeof(int32_t) * static_cast<size_t>(T) * k);          // row_of_slot
  n += align256(sizeof(int32_t) * R_cap) + align256(sizeof(float) * R_cap);
  n += align256(sizeof(float) * R_cap * gg_mx_rowdot_stride(F));        // rowdot
  n += align256(gg_workspace_size(T, k, E));
  return n;
}

gg_status gg_mx_buffers_bind(void* base, size_t bytes, int T, int H, int F, int k, int E,
                             int pad_multiple, gg_mx_buffers* out) {
  if (base == nullptr || out == nullptr) return GG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(base) & 255u) return GG_ERR_MISALIGNED;
  const size_t need = gg_mx_buffers_size(T, H, F, k, E, pad_multiple);
  if (need == 0) return GG_ERR_INVALID_ARG;
  if (bytes < need) return GG_ERR_WORKSPACE_TOO_SMALL;
  const size_t R_cap = static_cast<size_t>(r_cap_of(T, k, E, pad_multiple));
  const size_t nt = static_cast<size_t>(gg_mx_row_tiles(T, k, E, pad_multiple));
  const size_t h = static_cast<size_t>(H), f = static_cast<size_t>(F);
  uint8_t* p = static_cast<uint8_t*>(base);
  auto take = [&p](size_t n) {
    uint8_t* q = p;
    p += align256(n);
    return q;
  };
  std::memset(out, 0, sizeof(*out));
  out->Xq = take(R_cap * h);
  out->Xs = take(nt * (h / 128) * 512);
  out->dYq = take(R_cap * h);
  out->dYs = take(nt * (h / 128) * 512);
  out->Aq = take(R_cap * f);
  out->As = take(nt * (f / 128) * 512);
  out->dHq = take(R_cap * 2 * f);
  out->dHs = take(nt * (2 * f / 128) * 512);
  out->H1 = reinterpret_cast<gg_bf16*>(take(R_cap * 2 * f * 2));
  out->Yp = reinterpret_cast<gg_bf16*>(take(R_cap * h * 2));
  out->dXp = reinterpret_cast<gg_bf16*>(take(R_cap * h * 2));
  out->offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  out->tiles_before = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  out->row_of_slot =
      reinterpret_cast<int32_t*>(take(sizeof(int32_t) * static_cast<size_t>(T) * k));
  out->slot_of_row = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * R_cap));
  out->prob_of_row = reinterpret_cast<float*>(take(sizeof(float) * R_cap));
  out->rowdot = reinterpret_cast<float*>(take(sizeof(float) * R_cap * gg_mx_rowdot_stride(F)));
  out->n_tiles = static_cast<int>(nt);
  out->ws_bytes = align256(gg_workspace_size(T, k, E));
  out->ws = take(out->ws_bytes);
  return GG_OK;
}

static gg_status check_mx_buffers(const gg_mx_buffers* b, int T, int k, int E, int P) {
  if (b == nullptr) return GG_ERR_INVALID_ARG;
  if (b->Xq == nullptr || b->Xs == nullptr || b->H1 == nullptr || b->Aq == nullptr ||
      b->As == nullptr || b->Yp == nullptr || b->dYq == nullptr || b->dYs == nullptr ||
      b->dHq == nullptr || b->dHs == nullptr || b->dXp == nullptr || b->offsets == nullptr ||
      b->row_of_slot == nullptr || b->slot_of_row == nullptr || b->prob_of_row == nullptr ||
      b->tiles_before == nullptr || b->rowdot == nullptr)
    return GG_ERR_INVALID_ARG;
  if (b->n_tiles < gg_mx_row_tiles(T, k, E, P)) return GG_ERR_WORKSPACE_TOO_SMALL;
  return check_ws(b->ws, b->ws_bytes, gg_workspace_size(T, k, E));
}

static gg_status mx_layer_checks(int T, int H, int F, int k, int E, int P,
                                 const gg_moe_options* opt, const void* mxw,
                                 const gg_mx_buffers* buf, int* act, int* mode, int* R_cap) {
  if (T < 0 || k <= 0 || E <= 0 || P <= 0 || H <= 0 || F <= 0) return GG_ERR_INVALID_ARG;
  gg_epilogue fepi, bepi;
  bool recompute;
  gg_status s = read_options(opt, &fepi, &bepi, mode, &recompute);
  if (s != GG_OK) return s;
  if (recompute) return GG_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, H, F)) return GG_ERR_UNSUPPORTED_SHAPE;
  if ((s = check_mx_buffers(buf, T, k, E, P)) != GG_OK) return s;
  if (mxw == nullptr) return GG_ERR_INVALID_ARG;
  const long long rc = r_cap_of(T, k, E, P);
  if (rc > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  *R_cap = static_cast<int>(rc);
  *act = fepi == GG_EPI_QGEGLU ? GG_ACT_QGEGLU : GG_ACT_SWIGLU;
  return GG_OK;
}

gg_status gg_moe_mlp_fwd_mx(const gg_bf16* x, const int32_t* idx, const float* prob,
                            const void* mxw, int T, int H, int F, int k, int E,
                            int pad_multiple, const gg_moe_options* opt, gg_bf16* out,
                            const gg_mx_buffers* buf, gg_stream_t stream) {
  int act, mode, R_cap;
  gg_status s = mx_layer_checks(T, H, F, k, E, pad_multiple, opt, mxw, buf, &act, &mode, &R_cap);
  if (s != GG_OK) return s;
  if (T > 0 && (x == nullptr || out == nullptr)) return GG_ERR_INVALID_ARG;
  // row maps only: the permuted copy is the quantised one below
  s = gg_permute(x, idx, prob, T, H, k, E, pad_multiple, nullptr, buf->offsets, buf->row_of_slot,
                 buf->slot_of_row, buf->prob_of_row, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK || T == 0) return s;
  const bool pre = mode == GG_PROB_PRE_FC1;
  s = gg_mx_quantize_rows(x, T, H, k, buf->row_of_slot, buf->slot_of_row, buf->offsets,
                          pre ? prob : nullptr, E, pad_multiple, buf->n_tiles, buf->tiles_before,
                          buf->Xq, buf->Xs, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  s = gg_mx_grouped_gemm(GG_MX_FC1, act, buf->Xq, buf->Xs, mxw, buf->offsets, E, R_cap, H, F,
                         buf->n_tiles, nullptr, buf->Aq, buf->As, buf->H1,
                         mode == GG_PROB_ACTIVATION ? buf->prob_of_row : nullptr, nullptr,
                         buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  s = gg_mx_grouped_gemm(GG_MX_FC2, act, buf->Aq, buf->As, mxw, buf->offsets, E, R_cap, H, F,
                         buf->n_tiles, buf->Yp, nullptr, nullptr, nullptr, nullptr, nullptr,
                         buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  return gg_unpermute_combine(buf->Yp, buf->row_of_slot, mode == GG_PROB_COMBINE ? prob : nullptr,
                              T, k, H, R_cap, out, nullptr, 0, nullptr, nullptr, buf->ws,
                              buf->ws_bytes, stream);
}

gg_status gg_moe_mlp_bwd_mx(const gg_bf16* dOut, const gg_bf16* x, const float* prob,
                            const void* mxw, int T, int H, int F, int k, int E,
                            int pad_multiple, const gg_moe_options* opt, gg_bf16* dX,
                            float* dprob, const gg_mx_buffers* buf, gg_stream_t stream) {
  int act, mode, R_cap;
  gg_status s = mx_layer_checks(T, H, F, k, E, pad_multiple, opt, mxw, buf, &act, &mode, &R_cap);
  if (s != GG_OK) return s;
  if (T == 0) return GG_OK;
  if (dOut == nullptr || dX == nullptr) return GG_ERR_INVALID_ARG;
  const bool pre = mode == GG_PROB_PRE_FC1;
  if (pre && (prob == nullptr || (dprob != nullptr && x == nullptr))) return GG_ERR_INVALID_ARG;
  // Where the probability meets the forward decides where its gradient is
  // formed: at the combine (out = sum_j p * Yp, no quantiser in between) it
  // is <dOut_t, Yp[row]> on the kept Yp, formed in the dX combine; with the
  // weighted activation the probability sits inside FC2's quantised operand
  // and its gradient is the row sum of dA0 * act(H1), accumulated by the
  // SwiGLU-backward epilogue.
  float* rowdot = dprob != nullptr && mode == GG_PROB_ACTIVATION ? buf->rowdot : nullptr;
  s = gg_mx_quantize_rows(dOut, T, H, k, buf->row_of_slot, buf->slot_of_row, buf->offsets,
                          nullptr, E, pad_multiple, buf->n_tiles, buf->tiles_before, buf->dYq,
                          buf->dYs, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  s = gg_mx_grouped_gemm(GG_MX_DGRAD_FC2, act, buf->dYq, buf->dYs, mxw, buf->offsets, E, R_cap,
                         H, F, buf->n_tiles, nullptr, buf->dHq, buf->dHs, buf->H1,
                         pre ? nullptr : buf->prob_of_row, rowdot, buf->ws, buf->ws_bytes,
                         stream);
  if (s != GG_OK) return s;
  s = gg_mx_grouped_gemm(GG_MX_DGRAD_FC1, act, buf->dHq, buf->dHs, mxw, buf->offsets, E, R_cap,
                         H, F, buf->n_tiles, buf->dXp, nullptr, nullptr, nullptr, nullptr,
                         nullptr, buf->ws, buf->ws_bytes, stream);
  if (s != GG_OK) return s;
  if (pre)
    return gg_unpermute_combine(buf->dXp, buf->row_of_slot, prob, T, k, H, R_cap, dX, nullptr, 0,
                                dprob != nullptr ? x : nullptr, dprob, buf->ws, buf->ws_bytes,
                                stream);
  if (dprob != nullptr && mode == GG_PROB_COMBINE)
    return gg_unpermute_combine_dot(buf->dXp, buf->row_of_slot, nullptr, T, k, H, R_cap, dX,
                                    dOut, buf->Yp, dprob, buf->ws, buf->ws_bytes, stream);
  return gg_unpermute_combine(buf->dXp, buf->row_of_slot, nullptr, T, k, H, R_cap, dX, rowdot,
                              gg_mx_rowdot_blocks(F), nullptr, dprob, buf->ws, buf->ws_bytes,
                              stream);
}

gg_status gg_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                   gg_stream_t stream) {
  gg_status s = check_ws(ws, ws_bytes, kWsHeader);
  if (s != GG_OK) return s;
  DeviceInfo dev;
  if ((s = device_ok(&dev)) != GG_OK) return s;
  if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
  return from_cuda(launch_bounded_wait_selftest(status_ptr(ws), limit_ns,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
