// cfc_abi.cu -- extern "C" entry points of libcfc: argument validation on the host, per-device
// set-up (kernel attributes, cluster occupancy), launch planning and kernel launches.  The
// library allocates no memory and never synchronises (except cfc_device_status, whose purpose is
// to synchronise and read the status word).
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "cfc.h"
#include "cfc_kernels.h"

namespace cfc {
// Launcher of the failure-detection self-test kernel (cfc_selftest.cu).
cudaError_t wait_self_test_launch(int* status, cudaStream_t s);
// CTAs of the tau-decay BPTT launch for B rows (cfc_decay.cu).
int decay_bwd_ctas(int B);
}  // namespace cfc

namespace {

// Kernels record abandoned waits here; cfc_device_status reads and clears it.
__device__ int g_status_word;

struct DeviceState {
  bool init = false;
  int init_rc = CFC_OK;
  int sms = 0;
  int* status = nullptr;  // device address of g_status_word on this device
  std::map<std::tuple<int, int, int, size_t>, int> max_clusters;
};

constexpr int kMaxDevices = 64;
// Shared memory per CTA the launch plans assume (GB300's opt-in limit, 227 KB): plans, hence
// workspace sizes and summation orders, depend only on the problem sizes.
constexpr int kSmemBudget = 227 * 1024;
std::mutex g_mu;

bool valid_mode(int m) {
  return m == CFC_DW_ACCURATE || m == CFC_DW_BF16 || m == CFC_DW_TF32 || m == CFC_DW_SIMT_FP32;
}
// bf16 operand planes the BPTT writes for the contraction (0: fp32 d_pre).
int dpre_planes(int mode) {
  return mode == CFC_DW_ACCURATE ? 2 : mode == CFC_DW_BF16 ? 1 : 0;
}
DeviceState g_dev[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int cuda_rc(cudaError_t e, int code) {
  if (e == cudaSuccess) return CFC_OK;
  (void)cudaGetLastError();  // clear the sticky-free error so later calls are unaffected
  return code;
}

// Per-device initialisation under the lock; returns CFC_OK or an error code.
int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return CFC_ERR_UNSUPPORTED_DEVICE;
  }
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return CFC_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) {
      st.init = true;
      st.init_rc = CFC_ERR_UNSUPPORTED_DEVICE;
    } else {
      st.sms = sms;
      void* addr = nullptr;
      int rc = cuda_rc(cudaGetSymbolAddress(&addr, g_status_word), CFC_ERR_CUDA);
      if (rc == CFC_OK) rc = cuda_rc(cfc::reduce_axis0_prepare(), CFC_ERR_CUDA);
      int optin = 0;
      if (rc == CFC_OK)
        rc = cuda_rc(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                     CFC_ERR_CUDA);
      if (rc == CFC_OK) rc = cuda_rc(cfc::tc_prepare(optin), CFC_ERR_CUDA);
      if (rc == CFC_OK && optin < kSmemBudget) rc = CFC_ERR_UNSUPPORTED_DEVICE;
      if (rc == CFC_OK) rc = cuda_rc(cfc::contract_prepare(optin), CFC_ERR_CUDA);
      if (rc != CFC_OK) return rc;  // retried on the next call
      st.status = static_cast<int*>(addr);
      st.init = true;
      st.init_rc = CFC_OK;
    }
  }
  if (st.init_rc != CFC_OK) return st.init_rc;
  *out = &st;
  return CFC_OK;
}

// Smallest power of two >= ceil(C / channels per CTA): CTAs per cluster of a recurrence.
int cluster_size_for(int C, int chan_per_cta) {
  const int need = (C + chan_per_cta - 1) / chan_per_cta;
  int cs = 1;
  while (cs < need) cs <<= 1;
  return cs;
}

int check_dims(int B, int K, int C, int n_x) {
  if (B <= 0 || K <= 0 || C <= 0 || n_x <= 0) return CFC_ERR_INVALID_DIM;
  if (C > cfc::kMaxChannels) return CFC_ERR_INVALID_DIM;
  if (n_x > cfc::kMaxInputs) return CFC_ERR_INVALID_DIM;
  const long long pre = 4LL * K * B * C;
  if (pre >= (1LL << 31)) return CFC_ERR_INVALID_DIM;
  return CFC_OK;
}

// Cached cudaOccupancyMaxActiveClusters (prepare also sets the kernel attributes).
int max_clusters(DeviceState& st, int kind, int variant, int CS, size_t smem, int* out) {
  const auto key = std::make_tuple(kind, variant, CS, smem);
  auto it = st.max_clusters.find(key);
  if (it != st.max_clusters.end()) {
    *out = it->second;
    return CFC_OK;
  }
  int n = 0;
  // kind 0: forward (CUDA cores), 1: backward, 3 / 6: forward / backward with the tensor-core
  // contraction (`variant` is the rows per cluster, C = 32 CS)
  const cudaError_t e = (kind == 1)   ? cfc::bwd_prepare(CS, variant, smem, &n)
                       : (kind == 3) ? cfc::fwd_tc_prepare(CS * cfc::kFwdChanPerCta, variant, &n)
                       : (kind == 6) ? cfc::bwd_l2x_prepare(32 * CS, variant, &n)
                                     : cfc::fwd_prepare(CS, variant, smem, &n);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_CUDA;
  }
  st.max_clusters[key] = n;
  *out = n;
  return CFC_OK;
}

// Rows per cluster: the smallest R (power of two, <= 32) whose clusters all fit in one wave,
// else the largest that fits at all.  Results never depend on R (each row's arithmetic is the
// same whatever the grouping).
int plan_rows(DeviceState& st, int kind, int variant, int CS, int B, int n_x, int* R_out,
              size_t* smem_out, int* clusters_out, size_t min_smem = 0) {
  int best_R = 0;
  size_t best_smem = 0;
  const int r_max = (kind == 0) ? cfc::kMaxFwdRows : cfc::kMaxRowsPerCluster;
  for (int R = 1; R <= r_max; R *= 2) {
    size_t smem = (kind == 0) ? cfc::fwd_smem_bytes(R, CS) : cfc::bwd_smem_bytes(R, CS);
    if (smem < min_smem) smem = min_smem;
    int n = 0;
    // Each row count has its own kernel (and occupancy) up to four rows; the backward ring
    // kernel serves every larger count.
    const int kvar = (kind == 0 || R <= 4) ? R : 0;
    const int rc = max_clusters(st, kind, kvar, CS, smem, &n);
    if (rc != CFC_OK) return rc;
    if (n <= 0) break;
    best_R = R;
    best_smem = smem;
    if ((B + R - 1) / R <= n) break;
    if (R >= B) break;
  }
  if (best_R == 0) return CFC_ERR_INVALID_DIM;  // no cluster of this size can be scheduled
  *R_out = best_R;
  *smem_out = best_smem;
  *clusters_out = (B + best_R - 1) / best_R;
  return CFC_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct BwdLayout {
  size_t d_pre_off, d_pre_bytes;  // d_pre: fp32 rows, or the bf16 operand rows (4 mp bytes)
  size_t z_off, wt_off;           // contraction operands z [B*K] rows and W_u^T [n_x] rows
  size_t dt_off, zt_off;          // tf32: d_pre^T [4C][bkp] and z^T [n_in + 1][bkp] (fp32)
  size_t part_off, part_bytes;    // split partials of the weight-gradient contraction
  size_t total;
  int mp;                         // d_pre operand pitch
  int S_simt;                     // split count of the CUDA-core contraction
  cfc::ContractPlan pdw, pdu;     // tensor-core dW and du plans
  size_t pu_off;                  // du split partials (floats into the partials), if du is split
  bool tc_bptt;                   // the BPTT runs on the tensor cores (W_h^T pre-split at wsplit_off)
  size_t wsplit_off;
  size_t fwd_off;                 // cfc_forward_backward: the forward's workspace, last
};
// Rows (B*K) from which the input projection runs on the tensor cores (bf16 hi/lo split,
// tc_gemm_kernel<ProjProblem>) rather than on the CUDA cores (inproj_kernel): below it the
// CUDA-core kernel's single short wave is faster than the tensor-core kernel's set-up.
constexpr int kTcProjMinRows = 8192;

// Batch rows from which the forward recurrence runs its per-step gate contraction on the
// tensor cores (cfc_fwd_tc_kernel, 128 rows per cluster) instead of the CUDA-core kernel
// (at most 8 rows per cluster, one cluster per row group).  The tensor-core step time hardly
// grows with B, the CUDA-core one in steps of cluster waves; measured per step, C = 128: 5.3
// us (CUDA cores, B = 511) and 7.9 us (B = 767) against 7.6-7.7 us (tensor cores); C = 256:
// 11.8 us (CUDA cores, B <= 300) and 15.7 us (B = 400) against 12.2 us (tensor cores).
int tc_fwd_min_rows(int C) { return C >= 256 ? 384 : 768; }

// Workspace of the forward recurrence: the tensor-core kernel's exchange buffer, none for the
// CUDA-core kernel.
size_t fwd_ws_bytes(int B, int C) {
  return (B >= tc_fwd_min_rows(C) && cfc::fwd_tc_supported(C)) ? cfc::fwd_tc_xch_bytes(B, C) : 0;
}

// The tensor-core recurrence forms the input projection itself (one launch for the forward).
bool fwd_fused(int B, int C, int n_x) {
  return fwd_ws_bytes(B, C) > 0 && n_x <= cfc::kFwdFuseMaxInputs;
}

// CFC_OK when `ws` can hold the forward's workspace (nothing is needed below the tensor-core
// row threshold, and ws may then be NULL).
int check_fwd_ws(int B, int C, const void* ws, size_t ws_bytes) {
  const size_t need = fwd_ws_bytes(B, C);
  if (need == 0) return CFC_OK;
  if (!ws) return CFC_ERR_NULL_PTR;
  if (!aligned16(ws)) return CFC_ERR_MISALIGNED;
  return ws_bytes < need ? CFC_ERR_WS_TOO_SMALL : CFC_OK;
}

// Batch rows from which the BPTT recurrence runs its per-step contraction on the tensor cores
// (cfc_bwd_l2x_kernel, clusters of C / 32 CTAs per 128 or 144 rows); it needs the W_h^T image
// and the exchange blocks in the workspace.  Measured per step on GB300 (K = 32), C = 256: the
// CUDA-core kernel 9.7 us at B = 128 and 18.6 us at B = 256, the tensor-core one 10.2 us at
// either; C = 128: 7.6 us (CUDA cores, B = 512) and 14.5 us (B = 768) against 8.4-8.7 us.
int tc_bwd_min_rows(int C) { return C >= 256 ? 129 : 513; }

// Shared memory of a BPTT CTA launched as a dependent of the forward: more than half of an
// SM's 228 KB (so two BPTT CTAs cannot be packed onto one SM for the whole recurrence) and
// little enough to sit beside a forward CTA of 32 channels per CTA up to 128 channels.
constexpr size_t kDependentBwdSmem = 116 * 1024;

BwdLayout bwd_layout(int B, int K, int C, int n_x, int mode) {
  BwdLayout L{};
  const size_t BK = static_cast<size_t>(B) * K;
  const int n_in = n_x + C;
  L.d_pre_off = 0;
  if (mode == CFC_DW_SIMT_FP32) {
    L.mp = 4 * C;
    L.d_pre_bytes = BK * 4 * C * sizeof(float);
    L.S_simt = cfc::dw_simt_splits(static_cast<int>(BK));
    L.z_off = L.wt_off = L.part_off = align256(L.d_pre_bytes);
    L.part_bytes = static_cast<size_t>(L.S_simt) * 4 * C * n_in * sizeof(float);
  } else {
    const int form = mode;  // the tensor-core modes are the operand forms
    L.mp = cfc::contract_m_pitch(C, form);
    L.d_pre_bytes = BK * 4 * static_cast<size_t>(L.mp);  // 4 mp bytes per row in every form
    L.z_off = align256(L.d_pre_bytes);
    L.wt_off = align256(L.z_off + BK * 4 * static_cast<size_t>(cfc::contract_z_pitch(n_in, form)));
    L.part_off = align256(L.wt_off + static_cast<size_t>(n_x) * 4 * cfc::contract_wt_pitch(C));
    if (form == cfc::kFormTf32) {
      const size_t bkp = cfc::contract_bk_pitch(static_cast<int>(BK));
      L.dt_off = L.part_off;
      L.zt_off = align256(L.dt_off + static_cast<size_t>(4) * C * bkp * sizeof(float));
      L.part_off = align256(L.zt_off + static_cast<size_t>(n_in + 1) * bkp * sizeof(float));
    }
    cfc::contract_plans(B, K, C, n_x, form, kSmemBudget, &L.pdw, &L.pdu);
    L.pu_off = static_cast<size_t>(L.pdw.splits) * 4 * C * cfc::dw_tc_pitch(n_in);
    L.part_bytes = L.pu_off * sizeof(float);
    if (L.pdu.splits > 1) L.part_bytes += static_cast<size_t>(L.pdu.splits) * BK * n_x * sizeof(float);
  }
  L.total = L.part_off + L.part_bytes;
  L.tc_bptt = B >= tc_bwd_min_rows(C) && cfc::bwd_l2x_supported(C);
  L.wsplit_off = align256(L.total);
  if (L.tc_bptt) L.total = L.wsplit_off + cfc::bwd_l2x_ws_bytes(B, C);
  // Apart from everything the backward writes: the backward recurrence is a dependent launch
  // of the forward and may start while the forward still exchanges through it.
  L.fwd_off = align256(L.total);
  if (fwd_ws_bytes(B, C) > 0) L.total = L.fwd_off + fwd_ws_bytes(B, C);
  return L;
}

}  // namespace

extern "C" {

const char* cfc_error_string(int code) {
  switch (code) {
    case CFC_OK: return "ok";
    case CFC_ERR_INVALID_DIM: return "invalid or unsupported dimension";
    case CFC_ERR_NULL_PTR: return "required pointer is NULL";
    case CFC_ERR_MISALIGNED: return "tensor pointer is not 16-byte aligned";
    case CFC_ERR_WS_TOO_SMALL: return "workspace smaller than cfc_workspace_bytes()";
    case CFC_ERR_UNSUPPORTED_DEVICE: return "no usable compute capability 10.3 device";
    case CFC_ERR_LAUNCH_FAILED: return "kernel launch failed";
    case CFC_ERR_DEVICE_TIMEOUT: return "a kernel abandoned a bounded wait";
    case CFC_ERR_INVALID_ARG: return "invalid enumerated argument";
    case CFC_ERR_CUDA: return "CUDA runtime call failed";
    case CFC_ERR_SCRATCH_LIMIT:
      return "problem needs more workspace than cfc_backward_noalloc's built-in scratch holds";
    default: return "unknown status code";
  }
}

int cfc_workspace_bytes(int B, int K, int C, int n_x, int dw_mode, size_t* bwd_ws_bytes) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!valid_mode(dw_mode)) return CFC_ERR_INVALID_ARG;
  if (!bwd_ws_bytes) return CFC_ERR_NULL_PTR;
  *bwd_ws_bytes = bwd_layout(B, K, C, n_x, dw_mode).total;
  return CFC_OK;
}

int cfc_input_projection(const float* u, const float* W, const float* b, int B, int K, int C,
                         int n_x, float* H, float* cache, cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!u || !W || !b || !H || !cache) return CFC_ERR_NULL_PTR;
  if (!aligned16(u) || !aligned16(W) || !aligned16(b) || !aligned16(H) || !aligned16(cache))
    return CFC_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B * K >= kTcProjMinRows) {
    const cfc::TcPlan pl = cfc::proj_tc_plan(B, K, C, n_x);
    return cuda_rc(cfc::proj_tc_launch(pl, u, W, b, B, K, C, n_x, H, cache, st->status, s, false),
                   CFC_ERR_LAUNCH_FAILED);
  }
  return cuda_rc(cfc::inproj_launch(u, W, b, B * K, C, n_x, H, cache, s, false),
                 CFC_ERR_LAUNCH_FAILED);
}

}  // extern "C"

namespace {

// `pdl`: the previous kernel of the stream is one of this library's kernels of the same call
// (see cfc_launch.cuh).
// `xch`: the workspace of fwd_ws_bytes(B, C) bytes (checked by the caller; NULL when none is
// needed).  `u`, `b` (fused form, only where fwd_fused holds): the recurrence forms X = W_u u + b
// itself and nothing reads X from memory.
int forward_recurrence(const float* h0, const float* W, const float* ts, int B, int K, int C,
                       int n_x, float* H, float* cache, void* xch, cfc_stream_t stream, bool pdl,
                       const float* xH = nullptr, const float* xcache = nullptr,
                       bool out_bf16 = false, const float* u = nullptr,
                       const float* b = nullptr) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!h0 || !W || !ts || !H || !cache) return CFC_ERR_NULL_PTR;
  if (!aligned16(h0) || !aligned16(W) || !aligned16(ts) || !aligned16(H) || !aligned16(cache))
    return CFC_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  cfc::FwdParams p;
  p.u = nullptr; p.h0 = h0; p.W = W; p.bias = nullptr; p.ts = ts; p.H = H; p.cache = cache;
  p.xH = xH ? xH : H;  // X in place in H / cache unless given apart (bf16 outputs)
  p.xcache = xcache ? xcache : cache;
  p.out_bf16 = out_bf16 ? 1 : 0;
  p.status = st->status;
  p.B = B; p.K = K; p.C = C; p.n_x = n_x; p.n_in = n_x + C;
  p.CS = cluster_size_for(C, cfc::kFwdChanPerCta);
  p.xch = xch;
  const bool fuse = u && b;
  if (fwd_ws_bytes(B, C) > 0) {
    if (!xch) return CFC_ERR_NULL_PTR;
    // 128 rows per cluster, or 144 when 128-row clusters would not all be resident at once
    // (at C = 256, 2048 rows need 16 clusters of 8 CTAs and GB300 keeps 15: measured 21.3 us
    // per step in two waves against 12.2 us in one).
    int n = 0, n144 = 0;
    rc = max_clusters(*st, 3, 128, p.CS, 0, &n);
    if (rc != CFC_OK) return rc;
    p.R = 128;
    if (n > 0 && (B + 127) / 128 > n) {
      rc = max_clusters(*st, 3, 144, p.CS, 0, &n144);
      if (rc != CFC_OK) return rc;
      if (n144 > 0 && (B + 143) / 144 <= n144) p.R = 144;
    }
    if (n > 0) {
      if (fuse) {  // a non-NULL u asks the kernel for the fused form
        p.u = u;
        p.bias = b;
      }
      return cuda_rc(cfc::fwd_tc_launch(p, static_cast<cudaStream_t>(stream), pdl),
                     CFC_ERR_LAUNCH_FAILED);
    }
  }
  if (fuse) {
    // The tensor-core clusters cannot be scheduled: the CUDA-core recurrence reads X, which
    // the projection writes first (into H / cache; bf16 outputs have no room for it).
    if (out_bf16) return CFC_ERR_UNSUPPORTED_DEVICE;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B * K >= kTcProjMinRows) {
      const cfc::TcPlan pl = cfc::proj_tc_plan(B, K, C, n_x);
      rc = cuda_rc(cfc::proj_tc_launch(pl, u, W, b, B, K, C, n_x, H, cache, st->status, s, pdl),
                   CFC_ERR_LAUNCH_FAILED);
    } else {
      rc = cuda_rc(cfc::inproj_launch(u, W, b, B * K, C, n_x, H, cache, s, pdl),
                   CFC_ERR_LAUNCH_FAILED);
    }
    if (rc != CFC_OK) return rc;
    pdl = false;
  }
  size_t smem = 0;
  int n_clusters = 0;
  rc = plan_rows(*st, 0, 0, p.CS, B, n_x, &p.R, &smem, &n_clusters);
  if (rc != CFC_OK) return rc;
  return cuda_rc(cfc::fwd_launch(p, n_clusters, smem, static_cast<cudaStream_t>(stream), pdl),
                 CFC_ERR_LAUNCH_FAILED);
}

// The BPTT recurrence.  As a dependent launch (pdl) it may be scheduled while the previous
// kernel runs: it stages W_h^T and then waits for that kernel before it reads dH or the cache,
// so a dependent launch is only for a predecessor that writes neither W nor dH.  Its shared
// memory is then padded past half an SM, so that two BPTT CTAs never share one SM.
int backward_recurrence(const float* dH, const float* W, const float* ts, const float* cache,
                        int B, int K, int C, int n_x, float* d_pre, float* dh0,
                        cfc_stream_t stream, bool pdl, void* wsplit = nullptr, int dplanes = 0,
                        int dpitch = 0, bool cache_bf16 = false, int* free_sms = nullptr) {
  if (free_sms) *free_sms = 0;
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!dH || !W || !ts || !cache || !d_pre || !dh0) return CFC_ERR_NULL_PTR;
  if (!aligned16(dH) || !aligned16(W) || !aligned16(ts) || !aligned16(cache) ||
      !aligned16(d_pre) || !aligned16(dh0))
    return CFC_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  cfc::BwdParams p;
  p.dH = dH; p.W = W; p.ts = ts; p.cache = cache; p.d_pre = d_pre; p.dh0 = dh0;
  p.status = st->status;
  p.B = B; p.K = K; p.C = C; p.n_x = n_x; p.n_in = n_x + C;
  p.CS = cluster_size_for(C, cfc::kBwdChanPerCta);
  p.wsplit = wsplit;
  p.dplanes = dplanes;
  p.dpitch = dpitch;
  p.cache_bf16 = cache_bf16 ? 1 : 0;
  p.xbuf = nullptr;
  // The tensor-core BPTT moves dH, the cache and d_pre in whole 32-byte sectors.
  if (wsplit && B >= tc_bwd_min_rows(C) && cfc::bwd_l2x_supported(C) && aligned32(dH) &&
      aligned32(cache) && aligned32(d_pre)) {
    // Clusters of C / 32 CTAs per 128 rows when they are all resident at once, else per 144
    // rows (2048 rows: 15 clusters of 8 CTAs, the most GB300 keeps resident).
    int n128 = 0, n = 0;
    rc = max_clusters(*st, 6, 128, C / 32, 0, &n128);
    if (rc != CFC_OK) return rc;
    const int NR = cfc::bwd_l2x_rows(B, n128);
    rc = NR == 128 ? CFC_OK : max_clusters(*st, 6, NR, C / 32, 0, &n);
    if (rc != CFC_OK) return rc;
    if (NR == 128 || n > 0) {
      const cudaStream_t s = static_cast<cudaStream_t>(stream);
      rc = cuda_rc(cfc::bwd_l2x_split(W, C, n_x, wsplit, s, pdl), CFC_ERR_LAUNCH_FAILED);
      if (rc != CFC_OK) return rc;
      p.R = NR;
      p.xbuf = reinterpret_cast<float*>(static_cast<char*>(wsplit) + cfc::bwd_l2x_image_bytes(C));
      // SMs the recurrence leaves idle while every one of its clusters is resident.
      const int clusters = (B + NR - 1) / NR;
      if (free_sms && clusters <= (NR == 128 ? n128 : n))
        *free_sms = st->sms - clusters * (C / 32) > 0 ? st->sms - clusters * (C / 32) : 0;
      return cuda_rc(cfc::bwd_l2x_launch(p, NR, s, true), CFC_ERR_LAUNCH_FAILED);
    }
  }
  size_t smem = 0;
  int n_clusters = 0;
  rc = plan_rows(*st, 1, 0, p.CS, B, n_x, &p.R, &smem, &n_clusters,
                 pdl ? kDependentBwdSmem : 0);
  if (rc != CFC_OK) return rc;
  if (free_sms && st->sms > n_clusters * p.CS) *free_sms = st->sms - n_clusters * p.CS;
  return cuda_rc(cfc::bwd_launch(p, n_clusters, smem, static_cast<cudaStream_t>(stream), pdl),
                 CFC_ERR_LAUNCH_FAILED);
}

}  // namespace

extern "C" {

int cfc_forward_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!bytes) return CFC_ERR_NULL_PTR;
  *bytes = fwd_ws_bytes(B, C);
  return CFC_OK;
}

int cfc_forward_recurrence(const float* h0, const float* W, const float* ts, int B, int K,
                           int C, int n_x, float* H, float* cache, void* ws, size_t ws_bytes,
                           cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  rc = check_fwd_ws(B, C, ws, ws_bytes);
  if (rc != CFC_OK) return rc;
  return forward_recurrence(h0, W, ts, B, K, C, n_x, H, cache, ws, stream, false);
}

}  // extern "C"

namespace {
// cfc_forward after its argument checks; `xch` as for forward_recurrence.
int forward_all(const float* u, const float* h0, const float* W, const float* b,
                const float* ts, int B, int K, int C, int n_x, float* H, float* cache, void* xch,
                cfc_stream_t stream) {
  // Large batches: the tensor-core recurrence forms X itself (X never goes through memory:
  // at B = 2048, K = 128, C = 256 that is 1.07 GB written and read back).
  if (fwd_fused(B, C, n_x))
    return forward_recurrence(h0, W, ts, B, K, C, n_x, H, cache, xch, stream, false, nullptr,
                              nullptr, false, u, b);
  const int rc = cfc_input_projection(u, W, b, B, K, C, n_x, H, cache, stream);
  if (rc != CFC_OK) return rc;
  // Not a dependent launch: scheduled early, the recurrence clusters land on SMs the
  // projection still occupies and end up two CTAs to an SM, which slows every one of the K
  // steps (measured on GB300: the training step took 149.6 us this way against 140.7 us).
  return forward_recurrence(h0, W, ts, B, K, C, n_x, H, cache, xch, stream, false);
}
}  // namespace

extern "C" {

int cfc_forward(const float* u, const float* h0, const float* W, const float* b,
                const float* ts, int B, int K, int C, int n_x, float* H, float* cache, void* ws,
                size_t ws_bytes, cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!u || !h0 || !W || !b || !ts || !H || !cache) return CFC_ERR_NULL_PTR;
  if (!aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(b) || !aligned16(ts) ||
      !aligned16(H) || !aligned16(cache))
    return CFC_ERR_MISALIGNED;
  rc = check_fwd_ws(B, C, ws, ws_bytes);
  if (rc != CFC_OK) return rc;
  return forward_all(u, h0, W, b, ts, B, K, C, n_x, H, cache, ws, stream);
}

int cfc_step_launches(int B, int K, int C, int n_x, int dw_mode, int with_du, int* launches) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!valid_mode(dw_mode)) return CFC_ERR_INVALID_ARG;
  if (!launches) return CFC_ERR_NULL_PTR;
  // forward: projection + recurrence (the recurrence alone where it forms the projection
  // itself); backward: the recurrence (after the W_h^T pre-split on
  // the tensor-core path), then either the operand build, the dW contraction, du and the merge
  // (tensor-core modes), or the dW contraction, its merge, the db sum and du (CUDA cores).
  int n = (fwd_fused(B, C, n_x) ? 1 : 2) + 1 + 3 + (with_du ? 1 : 0);
  const BwdLayout L = bwd_layout(B, K, C, n_x, dw_mode);
  if (L.tc_bptt) n += 1;
  if (dw_mode == CFC_DW_TF32) n += 2;  // transposed copies of d_pre and z
  *launches = n;
  return CFC_OK;
}

int cfc_backward_recurrence(const float* dH, const float* W, const float* ts,
                            const float* cache, int B, int K, int C, int n_x, float* d_pre,
                            float* dh0, cfc_stream_t stream) {
  return backward_recurrence(dH, W, ts, cache, B, K, C, n_x, d_pre, dh0, stream, false);
}

int cfc_bptt_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!bytes) return CFC_ERR_NULL_PTR;
  *bytes = bwd_layout(B, K, C, n_x, CFC_DW_ACCURATE).tc_bptt ? cfc::bwd_l2x_ws_bytes(B, C) : 0;
  return CFC_OK;
}

int cfc_backward_recurrence_ws(const float* dH, const float* W, const float* ts,
                               const float* cache, int B, int K, int C, int n_x, float* d_pre,
                               float* dh0, void* ws, size_t ws_bytes, cfc_stream_t stream) {
  size_t need = 0;
  const int rc = cfc_bptt_workspace_bytes(B, K, C, n_x, &need);
  if (rc != CFC_OK) return rc;
  if (need > 0) {
    if (!ws) return CFC_ERR_NULL_PTR;
    if (!aligned16(ws)) return CFC_ERR_MISALIGNED;
    if (ws_bytes < need) return CFC_ERR_WS_TOO_SMALL;
  }
  return backward_recurrence(dH, W, ts, cache, B, K, C, n_x, d_pre, dh0, stream, false,
                             need > 0 ? ws : nullptr);
}

}  // extern "C"

namespace {

// The d_pre form the BPTT of cfc_backward writes: the contraction's operand rows, straight
// from either recurrence (fp32 rows for the TF32 and SIMT modes).  The tensor-core recurrence
// once wrote fp32 and a pass split it in place afterwards: 0.32 ms of HBM traffic at B=2048,
// K=128, C=256 that writing the rows directly does not cost.
int bptt_dplanes(const BwdLayout& /*L*/, int mode) { return dpre_planes(mode); }

// The standalone weight-gradient stage splits an fp32 d_pre into the workspace head.  That is
// safe when d_pre lies outside the head, or is the head itself with rows whose operand bytes
// are their fp32 bytes (each row is rewritten from its own values only); any other overlap is
// rejected.
struct BwdLayoutCheck {
  bool ok;
};
BwdLayoutCheck check_dpre_alias(const float* d_pre, bool dpre_in_ws, const char* head,
                                const BwdLayout& L, int B, int K, int C, int mode) {
  if (dpre_in_ws || mode == CFC_DW_SIMT_FP32 || mode == CFC_DW_TF32) return {true};
  const char* a = reinterpret_cast<const char*>(d_pre);
  const size_t a_bytes = static_cast<size_t>(B) * K * 4 * C * sizeof(float);
  const bool overlap = a < head + L.d_pre_bytes && head < a + a_bytes;
  if (!overlap) return {true};
  return {a == head && L.mp == 4 * C};
}

// `first_pdl`: the previous kernel of the stream is this library's BPTT recurrence of the same
// backward call; every later kernel here follows one of this function's own kernels.
// `dpre_in_ws`: d_pre is already in the workspace head in the mode's operand form (written so
// by the BPTT of cfc_backward); otherwise d_pre is fp32 [K][B][4][C] anywhere.
// `build_first`: the previous kernel is the BPTT recurrence, which releases its dependents only
// after its own dependency wait, so the operand build (which needs only the forward's outputs)
// runs beside it; otherwise the d_pre split comes first and the build runs beside that.
// `build_ctas` > 0: the build takes exactly that many CTAs (the SMs the recurrence leaves idle).
int weight_grad(const float* d_pre, const float* u, const float* h0, const float* W,
                const float* H, int B, int K, int C, int n_x, float* dW, float* db, float* du,
                void* ws, size_t ws_bytes, int dw_mode, cfc_stream_t stream, bool first_pdl,
                bool dpre_in_ws, bool build_first = false, bool h_bf16 = false,
                int build_ctas = 0) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!valid_mode(dw_mode)) return CFC_ERR_INVALID_ARG;
  if (!d_pre || !u || !h0 || !W || !H || !dW || !db || !ws) return CFC_ERR_NULL_PTR;
  if (!aligned16(d_pre) || !aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(H) ||
      !aligned16(dW) || !aligned16(db) || (du && !aligned16(du)) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(B, K, C, n_x, dw_mode);
  if (ws_bytes < L.total) return CFC_ERR_WS_TOO_SMALL;
  char* w = static_cast<char*>(ws);
  const BwdLayoutCheck chk = check_dpre_alias(d_pre, dpre_in_ws, w + L.d_pre_off, L, B, K, C,
                                              dw_mode);
  if (!chk.ok) return CFC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partial = reinterpret_cast<float*>(w + L.part_off);
  const int BK = B * K;
  const int M = 4 * C, N = n_x + C;
  if (dw_mode == CFC_DW_SIMT_FP32) {
    if (h_bf16) return CFC_ERR_INVALID_ARG;  // the CUDA-core contraction reads an fp32 H
    const int S = L.S_simt;
    rc = cuda_rc(cfc::dw_simt_launch(d_pre, u, H, h0, B, K, C, n_x, S, partial, s, first_pdl),
                 CFC_ERR_LAUNCH_FAILED);
    if (rc == CFC_OK)
      rc = cuda_rc(cfc::reduce_axis0_launch(partial, S, M * N, dW, s, true), CFC_ERR_LAUNCH_FAILED);
    if (rc == CFC_OK)
      rc = cuda_rc(cfc::reduce_axis0_launch(d_pre, BK, M, db, s, true), CFC_ERR_LAUNCH_FAILED);
    if (rc == CFC_OK && du)
      rc = cuda_rc(cfc::du_simt_launch(d_pre, W, BK, C, n_x, du, s, true), CFC_ERR_LAUNCH_FAILED);
    return rc;
  }
  // Tensor cores: the operand form is the mode.  The d_pre operand: the fp32 d_pre itself
  // (tf32), the rows the BPTT left in the workspace head, or a split of the fp32 d_pre into
  // the head (in place when d_pre is the head and a row's operand bytes are its fp32 bytes).
  const int form = dw_mode;
  const void* dop = form == cfc::kFormTf32 ? static_cast<const void*>(d_pre) : w + L.d_pre_off;
  const bool split = form != cfc::kFormTf32 && !dpre_in_ws;
  bool pdl = first_pdl;
  auto launch_build = [&]() {
    rc = cuda_rc(cfc::build_operands_launch(form, u, H, h_bf16 ? 1 : 0, h0, W, B, K, C, n_x,
                                            w + L.z_off, w + L.wt_off, s, pdl, 0, build_ctas),
                 CFC_ERR_LAUNCH_FAILED);
    pdl = true;
  };
  auto launch_split = [&]() {
    rc = cuda_rc(cfc::split_dpre_launch(form, d_pre, BK, C, w + L.d_pre_off, s, pdl),
                 CFC_ERR_LAUNCH_FAILED);
    pdl = true;
  };
  if (build_first || !split) {
    launch_build();
    if (rc == CFC_OK && split) launch_split();
  } else {
    launch_split();
    if (rc == CFC_OK) launch_build();
  }
  if (rc != CFC_OK) return rc;
  const void* a_dw = dop;
  const void* b_dw = w + L.z_off;
  if (form == cfc::kFormTf32) {
    // The tf32 weight gradient reads K-major copies: d_pre^T and z^T.
    const int bkp = cfc::contract_bk_pitch(BK);
    float* dt = reinterpret_cast<float*>(w + L.dt_off);
    float* zt = reinterpret_cast<float*>(w + L.zt_off);
    rc = cuda_rc(cfc::transpose_launch(d_pre, BK, M, M, dt, bkp, s, true), CFC_ERR_LAUNCH_FAILED);
    if (rc == CFC_OK)
      rc = cuda_rc(cfc::transpose_launch(reinterpret_cast<const float*>(w + L.z_off), BK, N + 1,
                                         cfc::contract_z_pitch(N, form), zt, bkp, s, true),
                   CFC_ERR_LAUNCH_FAILED);
    if (rc != CFC_OK) return rc;
    a_dw = dt;
    b_dw = zt;
  }
  const int pitch = cfc::dw_tc_pitch(N);
  rc = cuda_rc(cfc::dw_contract_launch(L.pdw, form, a_dw, b_dw, B, K, C, n_x, partial,
                                       pitch, st->status, s, true),
               CFC_ERR_LAUNCH_FAILED);
  if (rc != CFC_OK) return rc;
  float* du_out = (du && L.pdu.splits > 1) ? partial + L.pu_off : du;
  if (du) {
    rc = cuda_rc(cfc::du_contract_launch(L.pdu, form, dop, w + L.wt_off, B, K, C, n_x, du_out,
                                         st->status, s, true, true),
                 CFC_ERR_LAUNCH_FAILED);
    if (rc != CFC_OK) return rc;
  }
  // One merge: the dW partial rows carry the all-ones column, i.e. db; with split du, its
  // partials in the same launch.
  if (du && L.pdu.splits > 1)
    return cuda_rc(cfc::reduce_axis0_pair_launch(partial, L.pdw.splits, M * pitch, pitch, N, dW,
                                                 db, du_out, L.pdu.splits, BK * n_x, du, s, true),
                   CFC_ERR_LAUNCH_FAILED);
  return cuda_rc(cfc::reduce_axis0_rows_launch(partial, L.pdw.splits, M * pitch, pitch, N, dW, db,
                                               s, true),
                 CFC_ERR_LAUNCH_FAILED);
}

// The gradient stage right after the BPTT recurrence of the same call.  The operand build runs
// beside the recurrence on the SMs it leaves idle and nowhere else (1024-thread CTAs, which
// cannot share an SM with a recurrence CTA), so it never competes with the recurrence for issue
// slots.  With too few idle SMs it runs at its usual width: still beside the CUDA-core BPTT,
// after the tensor-core one (which holds most SMs).
constexpr int kMinBesideSms = 8;

int weight_grad_after_bptt(const float* d_pre, const float* u, const float* h0, const float* W,
                           const float* H, int B, int K, int C, int n_x, float* dW, float* db,
                           float* du, void* ws, size_t ws_bytes, int dw_mode,
                           cfc_stream_t stream, const BwdLayout& L, bool dpre_in_ws,
                           int free_sms, bool h_bf16) {
  const bool idle = free_sms >= kMinBesideSms;
  const bool beside = !L.tc_bptt || idle;
  return weight_grad(d_pre, u, h0, W, H, B, K, C, n_x, dW, db, du, ws, ws_bytes, dw_mode, stream,
                     beside, dpre_in_ws, beside, h_bf16, idle ? free_sms : 0);
}

}  // namespace

extern "C" {

int cfc_weight_grad(const float* d_pre, const float* u, const float* h0, const float* W,
                    const float* H, int B, int K, int C, int n_x, float* dW, float* db,
                    float* du, void* ws, size_t ws_bytes, int dw_mode, cfc_stream_t stream) {
  return weight_grad(d_pre, u, h0, W, H, B, K, C, n_x, dW, db, du, ws, ws_bytes, dw_mode,
                     stream, false, false);
}

int cfc_backward(const float* dH, const float* u, const float* h0, const float* W,
                 const float* ts, const float* H, const float* cache, int B, int K, int C,
                 int n_x, float* dW, float* db, float* du, float* dh0, void* ws,
                 size_t ws_bytes, int dw_mode, cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!valid_mode(dw_mode)) return CFC_ERR_INVALID_ARG;
  if (!dH || !u || !h0 || !W || !ts || !H || !cache || !dW || !db || !dh0 || !ws)
    return CFC_ERR_NULL_PTR;
  if (!aligned16(dH) || !aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(ts) ||
      !aligned16(H) || !aligned16(cache) || !aligned16(dW) || !aligned16(db) ||
      (du && !aligned16(du)) || !aligned16(dh0) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(B, K, C, n_x, dw_mode);
  if (ws_bytes < L.total) return CFC_ERR_WS_TOO_SMALL;
  float* d_pre = reinterpret_cast<float*>(static_cast<char*>(ws) + L.d_pre_off);
  const int dplanes = bptt_dplanes(L, dw_mode);
  int free_sms = 0;
  rc = backward_recurrence(dH, W, ts, cache, B, K, C, n_x, d_pre, dh0, stream, false,
                           L.tc_bptt ? static_cast<char*>(ws) + L.wsplit_off : nullptr, dplanes,
                           L.mp, false, &free_sms);
  if (rc != CFC_OK) return rc;
  return weight_grad_after_bptt(d_pre, u, h0, W, H, B, K, C, n_x, dW, db, du, ws, ws_bytes,
                                dw_mode, stream, L, dplanes == dpre_planes(dw_mode), free_sms,
                                false);
}

int cfc_forward_backward(const float* u, const float* h0, const float* W, const float* b,
                         const float* ts, const float* dH, int B, int K, int C, int n_x,
                         float* H, float* cache, float* dW, float* db, float* du, float* dh0,
                         void* ws, size_t ws_bytes, int dw_mode, cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!valid_mode(dw_mode)) return CFC_ERR_INVALID_ARG;
  if (!u || !h0 || !W || !b || !ts || !dH || !H || !cache || !dW || !db || !dh0 || !ws)
    return CFC_ERR_NULL_PTR;
  if (!aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(b) || !aligned16(ts) ||
      !aligned16(dH) || !aligned16(H) || !aligned16(cache) || !aligned16(dW) ||
      !aligned16(db) || (du && !aligned16(du)) || !aligned16(dh0) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(B, K, C, n_x, dw_mode);
  if (ws_bytes < L.total) return CFC_ERR_WS_TOO_SMALL;
  rc = forward_all(u, h0, W, b, ts, B, K, C, n_x, H, cache, static_cast<char*>(ws) + L.fwd_off,
                   stream);
  if (rc != CFC_OK) return rc;
  // The forward writes only H and cache, which the BPTT reads after its dependency wait.
  float* d_pre = reinterpret_cast<float*>(static_cast<char*>(ws) + L.d_pre_off);
  const int dplanes = bptt_dplanes(L, dw_mode);
  int free_sms = 0;
  rc = backward_recurrence(dH, W, ts, cache, B, K, C, n_x, d_pre, dh0, stream, true,
                           L.tc_bptt ? static_cast<char*>(ws) + L.wsplit_off : nullptr, dplanes,
                           L.mp, false, &free_sms);
  if (rc != CFC_OK) return rc;
  return weight_grad_after_bptt(d_pre, u, h0, W, H, B, K, C, n_x, dW, db, du, ws, ws_bytes,
                                dw_mode, stream, L, dplanes == dpre_planes(dw_mode), free_sms,
                                false);
}

// ---- bf16 state: H, the cache and d_pre stored as bf16, fp32 arithmetic ----

static size_t bf16_x_offset(int B, int K, int C) {
  return align256(static_cast<size_t>(K) * B * C * sizeof(float));
}

// After X (gate 0, then gates 1-3): the recurrence's own workspace.  The fused forward keeps
// no X: only that workspace.
static size_t bf16_xch_offset(int B, int K, int C, int n_x) {
  if (fwd_fused(B, C, n_x)) return 0;
  return align256(bf16_x_offset(B, K, C) + static_cast<size_t>(K) * B * 3 * C * sizeof(float));
}

int cfc_forward_bf16_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (C % 2 != 0) return CFC_ERR_INVALID_DIM;
  if (!bytes) return CFC_ERR_NULL_PTR;
  *bytes = bf16_xch_offset(B, K, C, n_x) + fwd_ws_bytes(B, C);
  return CFC_OK;
}

int cfc_forward_bf16(const float* u, const float* h0, const float* W, const float* b,
                     const float* ts, int B, int K, int C, int n_x, void* H, void* cache,
                     void* ws, size_t ws_bytes, cfc_stream_t stream) {
  size_t need = 0;
  int rc = cfc_forward_bf16_workspace_bytes(B, K, C, n_x, &need);
  if (rc != CFC_OK) return rc;
  if (!u || !h0 || !W || !b || !ts || !H || !cache || !ws) return CFC_ERR_NULL_PTR;
  if (!aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(b) || !aligned16(ts) ||
      !aligned16(H) || !aligned16(cache) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  if (ws_bytes < need) return CFC_ERR_WS_TOO_SMALL;
  if (fwd_fused(B, C, n_x))
    return forward_recurrence(h0, W, ts, B, K, C, n_x, static_cast<float*>(H),
                              static_cast<float*>(cache), ws, stream, false, nullptr, nullptr,
                              true, u, b);
  // X = W_u u + b in fp32, in the layouts of H and cache, in the workspace; then the
  // recurrence reads it there and stores H and the cache in bf16.
  float* xH = static_cast<float*>(ws);
  float* xcache = reinterpret_cast<float*>(static_cast<char*>(ws) + bf16_x_offset(B, K, C));
  rc = cfc_input_projection(u, W, b, B, K, C, n_x, xH, xcache, stream);
  if (rc != CFC_OK) return rc;
  return forward_recurrence(h0, W, ts, B, K, C, n_x, static_cast<float*>(H),
                            static_cast<float*>(cache),
                            static_cast<char*>(ws) + bf16_xch_offset(B, K, C, n_x), stream, false,
                            xH, xcache, true);
}

int cfc_backward_bf16(const float* dH, const float* u, const float* h0, const float* W,
                      const float* ts, const void* H, const void* cache, int B, int K, int C,
                      int n_x, float* dW, float* db, float* du, float* dh0, void* ws,
                      size_t ws_bytes, cfc_stream_t stream) {
  int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (C % 2 != 0) return CFC_ERR_INVALID_DIM;
  if (!dH || !u || !h0 || !W || !ts || !H || !cache || !dW || !db || !dh0 || !ws)
    return CFC_ERR_NULL_PTR;
  if (!aligned16(dH) || !aligned16(u) || !aligned16(h0) || !aligned16(W) || !aligned16(ts) ||
      !aligned16(H) || !aligned16(cache) || !aligned16(dW) || !aligned16(db) ||
      (du && !aligned16(du)) || !aligned16(dh0) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  const int mode = CFC_DW_BF16;  // d_pre in one bf16 plane, single-pass bf16 contractions
  const BwdLayout L = bwd_layout(B, K, C, n_x, mode);
  if (ws_bytes < L.total) return CFC_ERR_WS_TOO_SMALL;
  float* d_pre = reinterpret_cast<float*>(static_cast<char*>(ws) + L.d_pre_off);
  const int dplanes = bptt_dplanes(L, mode);
  int free_sms = 0;
  rc = backward_recurrence(dH, W, ts, static_cast<const float*>(cache), B, K, C, n_x, d_pre, dh0,
                           stream, false,
                           L.tc_bptt ? static_cast<char*>(ws) + L.wsplit_off : nullptr, dplanes,
                           L.mp, true, &free_sms);
  if (rc != CFC_OK) return rc;
  return weight_grad_after_bptt(d_pre, u, h0, W, static_cast<const float*>(H), B, K, C, n_x, dW,
                                db, du, ws, ws_bytes, mode, stream, L,
                                dplanes == dpre_planes(mode), free_sms, true);
}

int reduce_axis0(const float* per_batch, int n_batch, int n_tail, float* out,
                 cfc_stream_t stream) {
  if (n_batch <= 0 || n_tail <= 0) return CFC_ERR_INVALID_DIM;
  if (!per_batch || !out) return CFC_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(per_batch) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
    return CFC_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  return cuda_rc(cfc::reduce_axis0_launch(per_batch, n_batch, n_tail, out,
                                          static_cast<cudaStream_t>(stream), false),
                 CFC_ERR_LAUNCH_FAILED);
}

int cfc_wait_self_test(cfc_stream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  return cuda_rc(cfc::wait_self_test_launch(st->status, static_cast<cudaStream_t>(stream)),
                 CFC_ERR_LAUNCH_FAILED);
}

int cfc_device_status(int* status) {
  if (!status) return CFC_ERR_NULL_PTR;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_CUDA;
  }
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_CUDA;
  }
  *status = v;
  return CFC_OK;
}

}  // extern "C"

// ---- the pages' tau-decay cell ----

namespace {

// Backward workspace of the decay cell (offsets in bytes): da as bf16 operand rows, z rows,
// W_in^T rows, per-row dtau sums, then the contractions' split partials.
struct DecayLayout {
  int mp, zp, wp, ldo;
  size_t da_off, z_off, wt_off, dtau_off, part_off, pu_off, total;
  cfc::ContractPlan pdw, pdu;
};

DecayLayout decay_layout(int B, int K, int C, int n_x) {
  DecayLayout L{};
  const int form = cfc::kFormBf16x2;
  const size_t BK = static_cast<size_t>(B) * K;
  const int n_in = n_x + C;
  L.mp = (C + 7) & ~7;
  L.wp = L.mp;
  L.zp = cfc::contract_z_pitch(n_in, form);
  L.ldo = cfc::dw_tc_pitch(n_in);
  L.da_off = 0;
  L.z_off = align256(BK * 4 * L.mp);
  L.wt_off = align256(L.z_off + BK * 4 * L.zp);
  L.dtau_off = align256(L.wt_off + static_cast<size_t>(n_x) * 4 * L.wp);
  L.part_off = align256(L.dtau_off + static_cast<size_t>(B) * C * sizeof(float));
  cfc::contract_plans_mn(static_cast<int>(BK), C, n_in + 1, n_x, form, kSmemBudget, &L.pdw,
                         &L.pdu);
  L.pu_off = static_cast<size_t>(L.pdw.splits) * C * L.ldo;  // floats into the partials
  size_t part = L.pu_off * sizeof(float);
  if (L.pdu.splits > 1) part += static_cast<size_t>(L.pdu.splits) * BK * n_x * sizeof(float);
  L.total = L.part_off + part;
  return L;
}

int decay_check(int B, int K, int C, int n_x) {
  const int rc = check_dims(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!cfc::decay_supported(C, n_x)) return CFC_ERR_INVALID_DIM;
  return CFC_OK;
}

}  // namespace

extern "C" {

int cfc_decay_forward(const float* x, const float* h0, const float* W, const float* b,
                      const float* tau, const float* ts, int B, int K, int C, int n_x, float* H,
                      float* E, cfc_stream_t stream) {
  int rc = decay_check(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!x || !h0 || !W || !b || !tau || !ts || !H || !E) return CFC_ERR_NULL_PTR;
  if (!aligned16(x) || !aligned16(h0) || !aligned16(W) || !aligned16(b) || !aligned16(tau) ||
      !aligned16(ts) || !aligned16(H) || !aligned16(E))
    return CFC_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = cuda_rc(cfc::decay_proj_launch(x, W, b, B * K, C, n_x, E, s), CFC_ERR_LAUNCH_FAILED);
  if (rc != CFC_OK) return rc;
  return cuda_rc(cfc::decay_fwd_launch(h0, W, tau, ts, B, K, C, n_x, H, E, s),
                 CFC_ERR_LAUNCH_FAILED);
}

int cfc_decay_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes) {
  const int rc = decay_check(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!bytes) return CFC_ERR_NULL_PTR;
  *bytes = decay_layout(B, K, C, n_x).total;
  return CFC_OK;
}

int cfc_decay_backward(const float* dH, const float* x, const float* h0, const float* W,
                       const float* tau, const float* ts, const float* H, const float* E, int B,
                       int K, int C, int n_x, float* dW, float* db, float* dtau, float* dx,
                       float* dh0, void* ws, size_t ws_bytes, cfc_stream_t stream) {
  int rc = decay_check(B, K, C, n_x);
  if (rc != CFC_OK) return rc;
  if (!dH || !x || !h0 || !W || !tau || !ts || !H || !E || !dW || !db || !dtau || !dh0 || !ws)
    return CFC_ERR_NULL_PTR;
  if (!aligned16(dH) || !aligned16(x) || !aligned16(h0) || !aligned16(W) || !aligned16(tau) ||
      !aligned16(ts) || !aligned16(H) || !aligned16(E) || !aligned16(dW) || !aligned16(db) ||
      !aligned16(dtau) || (dx && !aligned16(dx)) || !aligned16(dh0) || !aligned16(ws))
    return CFC_ERR_MISALIGNED;
  const DecayLayout L = decay_layout(B, K, C, n_x);
  if (ws_bytes < L.total) return CFC_ERR_WS_TOO_SMALL;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != CFC_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const int form = cfc::kFormBf16x2;
  const int BK = B * K, n_in = n_x + C, N = n_in + 1;
  float* dtau_part = reinterpret_cast<float*>(w + L.dtau_off);
  float* partial = reinterpret_cast<float*>(w + L.part_off);
  // 1. BPTT: da straight into operand rows, dh0, per-row dtau sums.
  rc = cuda_rc(cfc::decay_bwd_launch(dH, h0, W, tau, ts, H, E, B, K, C, n_x, w + L.da_off, L.mp,
                                     dh0, dtau_part, s),
               CFC_ERR_LAUNCH_FAILED);
  // 2. z rows [x ; h_{t-1} ; 1] and W_in^T rows (W has C rows): beside the BPTT on the SMs it
  // leaves idle (1024-thread CTAs, which do not fit beside a BPTT CTA), else after it.
  const int idle = st->sms - cfc::decay_bwd_ctas(B);
  const bool beside = idle >= kMinBesideSms;
  if (rc == CFC_OK)
    rc = cuda_rc(cfc::build_operands_launch(form, x, H, 0, h0, W, B, K, C, n_x, w + L.z_off,
                                            w + L.wt_off, s, beside, C, beside ? idle : 0),
                 CFC_ERR_LAUNCH_FAILED);
  // 3. dW (with db in the ones column) and dx, one contraction each, dx beside dW.
  if (rc == CFC_OK)
    rc = cuda_rc(cfc::dw_contract_launch_mn(L.pdw, form, w + L.da_off, w + L.z_off, BK, C, N,
                                            L.mp, L.zp, partial, L.ldo, st->status, s, true),
                 CFC_ERR_LAUNCH_FAILED);
  float* dx_out = (dx && L.pdu.splits > 1) ? partial + L.pu_off : dx;
  if (rc == CFC_OK && dx)
    rc = cuda_rc(cfc::du_contract_launch_mn(L.pdu, form, w + L.da_off, w + L.wt_off, BK, C, n_x,
                                            L.mp, L.wp, dx_out, st->status, s, true, true),
                 CFC_ERR_LAUNCH_FAILED);
  // 4. One merge of the split partials, then dtau over the batch rows.
  if (rc == CFC_OK) {
    if (dx && L.pdu.splits > 1)
      rc = cuda_rc(cfc::reduce_axis0_pair_launch(partial, L.pdw.splits, C * L.ldo, L.ldo, n_in,
                                                 dW, db, dx_out, L.pdu.splits, BK * n_x, dx, s,
                                                 true),
                   CFC_ERR_LAUNCH_FAILED);
    else
      rc = cuda_rc(cfc::reduce_axis0_rows_launch(partial, L.pdw.splits, C * L.ldo, L.ldo, n_in,
                                                 dW, db, s, true),
                   CFC_ERR_LAUNCH_FAILED);
  }
  if (rc == CFC_OK)
    rc = cuda_rc(cfc::reduce_axis0_launch(dtau_part, B, C, dtau, s, true), CFC_ERR_LAUNCH_FAILED);
  return rc;
}

}  // extern "C"
