// cfc_kernels.h -- internal launch interface between the C-ABI entry points (cfc_abi.cu) and
// the kernels (one translation unit each).  Not part of the public header.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

namespace cfc {

// Channel tiling of the two recurrence kernels: every CTA of a cluster owns a fixed number of
// hidden channels (all four gates of each), so a cluster of CS CTAs covers that many x CS >= C.
constexpr int kFwdChanPerCta = 32;  // forward recurrence: a cluster of CS CTAs covers 32*CS
constexpr int kBwdChanPerCta = 32;  // backward recurrence, likewise
constexpr int kRecThreads = 256;
constexpr int kMaxClusterSize = 16;  // reduce_axis0 (non-portable clusters up to 16)
constexpr int kMaxChannels = 256;    // largest C: clusters of 8 CTAs x 32 channels
constexpr int kMaxInputs = 512;  // largest n_x (W_u rows of a CTA live in shared memory)
constexpr int kMaxRowsPerCluster = 32;  // backward recurrence
constexpr int kMaxFwdRows = 8;         // forward recurrence (rows are a template parameter)

struct FwdParams {
  // Set (with bias) only where the tensor-core recurrence forms X = W_u u + b itself
  // (n_x <= kFwdFuseMaxInputs); otherwise X is read from xH / xcache and u is NULL.
  const float* u;      // [K][B][n_x]
  const float* h0;     // [B][C]
  const float* W;      // [4][C][n_in]
  const float* bias;   // [4][C]
  const float* ts;     // [K][B]
  float* H;            // [K][B][C]              (bf16 elements when out_bf16)
  float* cache;        // [K][B][3][C]  (ff1, ff2, gate; bf16 elements when out_bf16)
  // X = W_u u + b in the layouts of H (gate 0) and cache (gates 1-3), fp32: the same arrays as
  // H / cache (written there in place by the projection) unless the outputs are bf16.
  const float* xH;
  const float* xcache;
  int out_bf16;        // H and cache are stored as bf16 (round to nearest even)
  int* status;         // device status word
  int B, K, C, n_x, n_in;
  int CS;              // CTAs per cluster
  int R;               // batch rows per cluster
  void* xch;           // tensor-core forward: the exchange buffer (fwd_tc_xch_bytes)
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
  const void* wsplit;  // tensor-core BPTT: the W_h^T image (bwd_l2x_split)
  // d_pre output form: 0 = fp32 [K][B][4][C] at d_pre; 1 or 2 = that many bf16 planes in the
  // contraction's operand rows (4 * dpitch bytes per row: hi, then lo) at d_pre.
  int dplanes;
  int dpitch;
  int cache_bf16;      // the cache holds bf16 elements
  float* xbuf;         // bwd_l2x_launch: the clusters' exchange blocks (bwd_l2x_ws_bytes)
};

// Every launch function takes `pdl`: schedule the kernel while the previous kernel of the
// stream is still running (programmatic dependent launch; see cfc_launch.cuh).  Set only
// between two kernels of the same entry point.

// Recurrence kernels (persistent over all K steps, one cluster per group of R batch rows).
size_t fwd_smem_bytes(int R, int CS);
cudaError_t fwd_prepare(int CS, int R, size_t smem, int* max_active_clusters);
cudaError_t fwd_launch(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
                       bool pdl);

// The forward recurrence with each step's gate contraction on the tensor cores (clusters of
// C / 32 CTAs serving 128 or 144 batch rows each, FwdParams::R; C = 128 or 256).  X in place
// in H / cache as for fwd_launch.
bool fwd_tc_supported(int C);
// Inputs up to which the tensor-core forward can form the input projection itself.
constexpr int kFwdFuseMaxInputs = 64;
cudaError_t fwd_tc_prepare(int C, int rows, int* max_active_clusters);
cudaError_t fwd_tc_launch(const FwdParams& p, cudaStream_t s, bool pdl);
// Bytes of the tensor-core forward's exchange buffer for B rows (either row tile), 16-byte
// aligned slots.
size_t fwd_tc_xch_bytes(int B, int C);

// The BPTT recurrence with each step's contraction split along its reduction over a cluster of
// C / 32 CTAs per NR = 128 or 144 batch rows (rows along the MMA's N side, C = 128 or 256), the
// partial sums exchanged through L2.  Workspace (bwd_l2x_ws_bytes): the W_h^T image written by
// bwd_l2x_split (bwd_l2x_image_bytes), then the exchange blocks (BwdParams::xbuf).  Writes fp32
// d_pre.  bwd_l2x_rows: 128 when ceil(B / 128) clusters of that tile are resident at once.
bool bwd_l2x_supported(int C);
int bwd_l2x_rows(int B, int max_clusters_128);
size_t bwd_l2x_image_bytes(int C);
size_t bwd_l2x_ws_bytes(int B, int C);
cudaError_t bwd_l2x_prepare(int C, int NR, int* max_active_clusters);
cudaError_t bwd_l2x_split(const float* W, int C, int n_x, void* ws, cudaStream_t s, bool pdl);
cudaError_t bwd_l2x_launch(const BwdParams& p, int NR, cudaStream_t s, bool pdl);

size_t bwd_smem_bytes(int R, int CS);
cudaError_t bwd_prepare(int CS, int R, size_t smem, int* max_active_clusters);
cudaError_t bwd_launch(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
                       bool pdl);

// X = W_u u + b for all steps, written in place into H (gate ff1) and cache (ff2, ta, tb).
cudaError_t inproj_launch(const float* u, const float* W, const float* bias, int BK, int C,
                          int n_x, float* H, float* cache, cudaStream_t s, bool pdl);

// Weight gradient, split over the B*K reduction: partial[s][m][n] for m < 4C, n < n_in.
int dw_simt_splits(int BK);
cudaError_t dw_simt_launch(const float* d_pre, const float* u, const float* H, const float* h0,
                           int B, int K, int C, int n_x, int S, float* partial, cudaStream_t s,
                           bool pdl);

// The input projection X = W_u u + b on the tensor cores (three bf16 terms per operand, six
// products), written in place into H and cache like inproj_launch.
struct TcPlan {
  int n_tiles, n_tile, m_tiles, n_kb, kb_per_split, splits;
  int mt;  // 128-row accumulators per CTA
  size_t smem;
};
cudaError_t tc_prepare(int max_smem);
TcPlan proj_tc_plan(int B, int K, int C, int n_x);
cudaError_t proj_tc_launch(const TcPlan& pl, const float* u, const float* W, const float* bias,
                           int B, int K, int C, int n_x, float* H, float* cache, int* status,
                           cudaStream_t s, bool pdl);

// ---- TMA-fed contractions (cfc_contract.cu) ----
// Operand forms of the backward contractions, one per tensor-core weight-gradient mode.
constexpr int kFormBf16x2 = 0;  // two bf16 planes, hi and lo: three MMAs per step (accurate)
constexpr int kFormBf16 = 1;    // the hi plane alone: one MMA per step
constexpr int kFormTf32 = 2;    // the fp32 values: one kind::tf32 MMA per step
// Operand layout: row r of an operand occupies 4 * pitch bytes.  bf16 forms: the hi plane's
// `pitch` values, then the lo plane's (unused in the bf16 form); tf32: `pitch` floats.  With
// pitch = 4C a d_pre row has exactly the bytes of its fp32 row.
int contract_m_pitch(int C, int form);     // d_pre rows: >= 4C (exactly 4C for tf32)
int contract_wt_pitch(int C);              // W_u^T rows: >= 4C
int contract_bk_pitch(int BK);             // tf32 transposed operands: rows of >= B*K floats
// dst[c][r] = src[r][c] (fp32; rows sp / dp floats apart).
cudaError_t transpose_launch(const float* src, int rows, int cols, int sp, float* dst, int dp,
                             cudaStream_t s, bool pdl);
int contract_z_pitch(int n_in, int form);  // z rows: >= n_in + 1

struct ContractPlan {
  int mt;       // 128-row accumulators per CTA
  int n_tile, n_tiles, m_tiles;
  int n_kb, kb_per_split, splits;
  int kd;       // reduction entries per k-block
  int stages;
  size_t smem;
};
ContractPlan dw_contract_plan(int B, int K, int C, int n_x, int form, int smem_budget);
ContractPlan du_contract_plan(int B, int K, int C, int n_x, int form, int smem_budget);
// Both plans as the backward pass uses them: for small B*K both are split, sized together so
// their CTAs fill one wave (du then writes split partials [splits][B*K][n_x]).
void contract_plans(int B, int K, int C, int n_x, int form, int smem_budget, ContractPlan* pw,
                    ContractPlan* pu);
// The same with the sizes explicit (the four-gate cell: M = 4C gate rows, N = n_x + C + 1 z
// columns; the decay cell: M = C): d_pre [BK][M], z [BK][N], W_u^T [n_x][M].
ContractPlan dw_contract_plan_mn(int BK, int M, int N, int form, int smem_budget);
ContractPlan du_contract_plan_mn(int BK, int M, int n_x, int form, int smem_budget);
void contract_plans_mn(int BK, int M, int N, int n_x, int form, int smem_budget,
                       ContractPlan* pw, ContractPlan* pu);
cudaError_t contract_prepare(int max_smem);
// z rows [u ; h_{t-1} ; 1] (B*K of them) and W_u^T rows (n_x) in the operand form; H is fp32,
// or bf16 when h_bf16.  W has M rows of n_x + C (M <= 0: 4C, the four gates); W_u^T rows are
// (M + 7) & ~7 values apart.  `ctas` > 0: exactly that many CTAs of 1024 threads, for a build
// that runs on the SMs a concurrent kernel leaves idle; otherwise a grid-stride launch of up
// to two 256-thread CTAs per SM.
cudaError_t build_operands_launch(int form, const float* u, const void* H, int h_bf16,
                                  const float* h0, const float* W, int B, int K, int C, int n_x,
                                  void* z, void* wt, cudaStream_t s, bool pdl, int M = 0,
                                  int ctas = 0);
// fp32 d_pre [B*K][4C] -> the bf16 operand rows (may be in place when the pitch is 4C).
cudaError_t split_dpre_launch(int form, const float* d_pre, int BK, int C, void* planes,
                              cudaStream_t s, bool pdl);
// dW partials [splits][4C][ldo] (column n_in is db) from the d_pre operand and z.
cudaError_t dw_contract_launch(const ContractPlan& pl, int form, const void* dpre, const void* z,
                               int B, int K, int C, int n_x, float* partial, int ldo,
                               int* status, cudaStream_t s, bool pdl);
// du [B*K][n_x] (or, when the plan splits, partials [splits][B*K][n_x]) from the d_pre operand
// and W_u^T.  `defer_wait`: launched right after the
// weight-gradient contraction of the same call, whose operands it shares; it then runs beside
// that kernel and waits for it only at its end.
cudaError_t du_contract_launch(const ContractPlan& pl, int form, const void* dpre, const void* wt,
                               int B, int K, int C, int n_x, float* du, int* status,
                               cudaStream_t s, bool pdl, bool defer_wait);
// The two contractions with the sizes and operand pitches explicit (mp: d_pre rows, zp: z
// rows, wp: W_u^T rows; 4 * pitch bytes per row).
cudaError_t dw_contract_launch_mn(const ContractPlan& pl, int form, const void* dpre,
                                  const void* z, int BK, int M, int N, int mp, int zp,
                                  float* partial, int ldo, int* status, cudaStream_t s, bool pdl);
cudaError_t du_contract_launch_mn(const ContractPlan& pl, int form, const void* dpre,
                                  const void* wt, int BK, int M, int n_x, int mp, int wp,
                                  float* du, int* status, cudaStream_t s, bool pdl,
                                  bool defer_wait);

// du[r][k] = sum_m d_pre[r][m] * W[m][k] for k < n_x (SIMT fp32).
cudaError_t du_simt_launch(const float* d_pre, const float* W, int BK, int C, int n_x,
                           float* du, cudaStream_t s, bool pdl);

// Deterministic axis-0 sum with overwrite semantics.
cudaError_t reduce_axis0_prepare();
cudaError_t reduce_axis0_launch(const float* in, int n_batch, int n_tail, float* out,
                                cudaStream_t s, bool pdl);
// The same sum over a tail of rows of `pitch` values: columns < ncol of each row go to
// out[row][ncol], column ncol to out2[row], the rest (padding) is dropped.
cudaError_t reduce_axis0_rows_launch(const float* in, int n_batch, int n_tail, int pitch,
                                     int ncol, float* out, float* out2, cudaStream_t s,
                                     bool pdl);
// Two such sums in one launch: (in, n_batch, n_tail, pitch, ncol -> out, out2) as
// reduce_axis0_rows_launch, and (in_b, n_batch_b, n_tail_b -> out_b) as reduce_axis0_launch.
cudaError_t reduce_axis0_pair_launch(const float* in, int n_batch, int n_tail, int pitch,
                                     int ncol, float* out, float* out2, const float* in_b,
                                     int n_batch_b, int n_tail_b, float* out_b, cudaStream_t s,
                                     bool pdl);
// The pages' tau-decay cell (cfc_decay.cu): hidden width at most kDecayMaxC.
constexpr int kDecayMaxC = 128;
bool decay_supported(int C, int n_x);
// X = W_in x + b for the B*K rows, into E [B*K][C].
cudaError_t decay_proj_launch(const float* x, const float* W, const float* b, int BK, int C,
                              int n_x, float* E, cudaStream_t s);
// The K-step recurrence reading X from E and writing H and E = tanh(a).
cudaError_t decay_fwd_launch(const float* h0, const float* W, const float* tau, const float* ts,
                             int B, int K, int C, int n_x, float* H, float* E, cudaStream_t s);
// BPTT: da as bf16 operand rows (2 mp values per row, hi then lo), dh0, per-row dtau sums.
cudaError_t decay_bwd_launch(const float* dH, const float* h0, const float* W, const float* tau,
                             const float* ts, const float* H, const float* E, int B, int K,
                             int C, int n_x, void* da_rows, int mp, float* dh0, float* dtau_part,
                             cudaStream_t s);

// Row pitch of the tensor-core weight-gradient partials: the n_in columns of z, the all-ones
// column that yields db, padded to a multiple of 4.
inline int dw_tc_pitch(int n_in) { return (n_in + 1 + 3) & ~3; }

}  // namespace cfc
