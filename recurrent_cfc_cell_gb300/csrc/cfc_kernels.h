// cfc_kernels.h -- internal launch interface between the C-ABI entry points (cfc_abi.cu) and
// the kernels (one translation unit each).  Not part of the public header.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

namespace cfc {

// Channel tiling shared by the two recurrence kernels: every CTA of a cluster owns 16 hidden
// channels (all four gates of each), so a cluster of CS CTAs covers 16*CS >= C channels.
constexpr int kChanPerCta = 16;
constexpr int kRowsPerCta = 4 * kChanPerCta;  // W rows held by one CTA (gate-minor order)
constexpr int kRecThreads = 256;
constexpr int kMaxClusterSize = 16;
constexpr int kMaxZ = 320;      // padded z width the forward kernel holds in registers
constexpr int kMaxRowsPerCluster = 32;

struct FwdParams {
  const float* u;      // [K][B][n_x]
  const float* h0;     // [B][C]
  const float* W;      // [4][C][n_in]
  const float* bias;   // [4][C]
  const float* ts;     // [K][B]
  float* H;            // [K][B][C]
  float* cache;        // [K][B][3][C]  (ff1, ff2, gate)
  int* status;         // device status word
  int B, K, C, n_x, n_in;
  int CS;              // CTAs per cluster
  int R;               // batch rows per cluster
  int nxp;             // n_x rounded up to a multiple of 4
  int NZp;             // padded z width (4 slices x KW)
};

struct BwdParams {
  const float* dH;     // [K][B][C]
  const float* W;      // [4][C][n_in]
  const float* ts;     // [K][B]
  const float* cache;  // [K][B][3][C]
  float* d_pre;        // [K][B][4][C]
  float* dh0;          // [B][C]
  int* status;
  int B, K, C, n_x, n_in;
  int CS, R;
};

// Recurrence kernels (persistent over all K steps, one cluster per group of R batch rows).
int fwd_kw_for(int nxp, int CS);  // register width per K-slice, or -1 if unsupported
size_t fwd_smem_bytes(int R, int NZp);
cudaError_t fwd_prepare(int KW, int CS, size_t smem, int* max_active_clusters);
cudaError_t fwd_launch(int KW, const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s);

size_t bwd_smem_bytes(int R);
cudaError_t bwd_prepare(int CS, size_t smem, int* max_active_clusters);
cudaError_t bwd_launch(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s);

// Weight gradient, split over the B*K reduction: partial[s][m][n] for m < 4C, n < n_in.
int dw_simt_splits(int BK);
cudaError_t dw_simt_launch(const float* d_pre, const float* u, const float* H, const float* h0,
                           int B, int K, int C, int n_x, int S, float* partial, cudaStream_t s);

// du[r][k] = sum_m d_pre[r][m] * W[m][k] for k < n_x (SIMT fp32).
cudaError_t du_simt_launch(const float* d_pre, const float* W, int BK, int C, int n_x,
                           float* du, cudaStream_t s);

// Deterministic axis-0 sum with overwrite semantics.
cudaError_t reduce_axis0_prepare();
cudaError_t reduce_axis0_launch(const float* in, int n_batch, int n_tail, float* out,
                                cudaStream_t s);

}  // namespace cfc
