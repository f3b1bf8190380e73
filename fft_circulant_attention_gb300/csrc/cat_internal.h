// Internal plan structure and kernel launchers of libcat (not part of the ABI).
#pragma once
#include <cstdlib>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "fft_device.cuh"

namespace cat {

enum Path { PATH_SMEM = 0, PATH_FOURSTEP = 1, PATH_FAST = 2, PATH_DIRECT = 3 };

// Launch shape of the single-CTA shared-memory path (N up to 16384): one CTA
// transforms G packed column pairs of one (b, h).
struct SmemCfg {
  int G;             // column pairs per CTA
  int groups;        // CTAs per (b, h) = ceil(npair / G)
  int tstride;       // shared-memory stride between transforms (complex)
  int threads;       // CTA size of the conv kernel
  size_t smem;       // dynamic shared memory of the conv kernel (bytes)
  int spec_threads;  // CTA size of the softmax+spectrum kernel
  size_t spec_smem;
  int reg_m;         // N = reg_m² transformed in registers (conv_reg), else 0
};

// Launch shape of the direct (O(N²·dh), no transform) path for short
// sequences: one CTA of threads = (dh/4)·nrg per (R-row tile, b, h); thread
// (rg, cg) owns TR rows and 4 columns.  fused: the CTA computes its row's
// scores from X and W_A itself (the whole forward is one launch).
struct DirectCfg {
  int TR, nrg, R, threads, fused;
  size_t smem;
};

// 2-D plan on a square grid of side M = 32·R (64, 96, 128): the five-pass
// row/column transform of grid_pass.cu over chunks of `chunk` (b, h) rows.
struct GridPassCfg {
  int M, R, chunk;
  size_t scratch_bytes;
};

// Four-step decomposition N = N1·N2 with row n = n1 + N1·n2 and bin
// k = N2·k1 + k2.  Column pass A: per n1, DFT over n2 (length N2), then the
// twiddle exp(-2πi n1·k2/N).  Row pass B: per k2, DFT over n1 (length N1),
// product with the spectrum of z*, inverse DFT back to n1, conjugate
// twiddle.  Column pass C: per n1, inverse DFT over k2 back to n2.
// Scratch row layout per (b, h): [k2][n1][P] complex, P = npair + 1 signals
// (the last one carries z* through pass A).
struct FourStepCfg {
  int N1, N2;
  RadixPlan rp1, rp2;   // radices of N1 (pass B) and N2 (passes A, C)
  int G, groups;        // pairs per CTA, CTAs per (b, h) along the pairs
  int TA;               // n1 values per CTA in passes A and C (divides N1)
  int TB;               // k2 values per CTA in pass B (divides N2)
  int P;                // signals per scratch row = npair + 1
  int threadsA, threadsB, threadsC;
  size_t smemA, smemB, smemC;
  int chunk_bh;         // (b, h) rows whose scratch is live at once
  int a_tma_per_sm;     // fast path, N2 > 32: resident CTAs per SM of the
                        // tensor-copy pass A (0: the plain pass A)
};

// Backward correlation dz*[k] = sum_c sum_i G[i, c] V[(i - k) mod N, c] by
// the four-step split N = N1·N2 (N1 = N, N2 = 1 for short rows).  Scratch
// row layout per (b, h): [k2][n1][Q] complex, Q = 2·npair signals (G pairs,
// then V pairs); signal 0 receives the correlation's partial inverse.
struct BwCfg {
  int N1, N2;
  RadixPlan rp1, rp2;
  int GA, groupsA, TA, threadsA;   // pass A: pairs per CTA, CTAs per (b, h), n1 per CTA
  size_t smemA;
  int GB, TB, threadsB;            // pass B: pairs per chunk, k2 per CTA
  size_t smemB;
  int TC, threadsC;                // pass C: n1 per CTA
  size_t smemC;
  int fast;                        // 1: the fast path's passes A and fsf_corr_b
  int Q;                           // scratch signals per (b, h) = 2·npair (fast: 1)
  int chunk_bh;                    // (b, h) rows whose scratch is live at once
  int wsplit;                      // token ranges of the dW_A partial sums
  size_t scratch_bytes;
};

}  // namespace cat

struct cat_plan_s {
  CUtensorMap tm_c[2];      // fast path: scratch views for pass C (TMA), per slot
  int B, N, D, H, dtype;
  int dh, npair;            // head width, packed pairs per head = ceil(dh/2)
  int device;
  int sms;                  // multiprocessors of the device
  cudaStream_t stream;
  int path;
  cat::RadixPlan rpN;       // radices of N (shared-memory path)
  cat::SmemCfg sm;
  cat::FourStepCfg fs;
  cat::DirectCfg dir;
  int score_cuda_cores;     // 1: bf16 scores on the CUDA-core kernel (testing)
  int score_path;           // 1: bf16 scores on the register-fed MMA kernel (testing)
  int fork_at;              // fast path: where the chunk streams fork (cat::FORK_*)
  int fast_pdl;             // fast path: passes launched as programmatic dependents of
                            // the pass ahead on their stream (0 no, 1 signal at the
                            // end of each CTA, 2 at its start)
  // workspace (device)
  float2* z2;               // [B, H, N] scores as double-float (hi, lo)
  float* zs;                // [B, H, N] z* (softmax weights)
  float2* part;             // [B, H, P] softmax partials (max, sum) per chunk
  float2* zf;               // [B, H, N] spectrum of z* divided by N (smem path)
  float2* tw;               // [N] exp(-2πi j/N)
  float2* zscr;             // [B, H, N] fast path: z* after its first DFT pass
  float2* tabs;             // fast path: pass-B twiddle tables
  float2* scratch;          // four-step scratch, chunk_bh·N·P complex (fast path: 2 slots)
  size_t scratch_bytes;
  // fast path: two internal streams that run alternate batches / chunks so
  // that one's score and small kernels overlap the other's FFT passes
  cudaStream_t side[2];
  cudaEvent_t ev_fork, ev_join[2], ev_front[2];
  // fast path: the overlapped schedule captured once as a CUDA graph (on the
  // private stream cap) and replayed while the call's pointers stay the same
  int use_graph;
  cudaStream_t cap;
  cudaGraphExec_t gexec;
  const void* gX; const void* gWA; const void* gV; void* gO;
  // fast path: the backward's schedule captured the same way (its own graph;
  // the pointers it was captured with)
  cudaGraphExec_t bgexec;
  const void* bgp[7];
  unsigned int* status;     // device status word
  size_t workspace_bytes;
  // host-buffer calls (cat_forward_host), set up at the first such call:
  // device staging (two slots of one batch each when B >= 2, else one slot
  // of the whole problem), two one-batch sub-plans that alternate between the
  // slots, the copy streams (0: host to device, 1: device to host) and the
  // events that order a slot's copies and compute
  int hready;
  void* hx[2]; void* hv[2]; void* ho[2]; void* hwa;
  cat_plan_s* hsub[2];
  cudaStream_t hcp[2];
  cudaEvent_t hev_in[2], hev_done[2], hev_out[2];
  // fused projection (cat_forward_fused): the K-major B operands W_V^T and
  // W_A^T, allocated at the first such call
  void* pj_wt;
  // stage timing: 4 events per recorded call (before score, after score,
  // after softmax/spectrum, after the circulant product)
  cudaEvent_t* ev;
  int timing_cap, timing_n;
  int ev_per_call;          // events recorded per call (3 + conv pass boundaries)
  int launches;             // kernel launches per cat_forward
  // 2-D plan (cat_plan_create_2d): tokens on a grid_h x grid_w grid, the
  // generic four-step passes without twiddles (N1 = grid_w, N2 = grid_h)
  int twod, grid_h, grid_w;
  // 2-D plan on a square grid of side 8, 14, 16 or 32: the register kernels
  // without twiddles (scores, spectrum, product) instead of the generic passes
  int reg2d;
  // 2-D plan on a square grid of side 64, 96 or 128: the row/column passes
  // of grid_pass.cu (scratch: p->scratch)
  int gp2d;
  cat::GridPassCfg gp;
  // backward workspace (configured and allocated at the first backward call)
  int bw_ready;
  cat::BwCfg bw;
  float2* bw_scr;           // correlation scratch, chunk_bh·N·Q complex
  float* bw_dzs;            // [B, H, N] dL/dz*
  float* bw_dz;             // [B, H, N] dL/dz
  float* bw_wpart;          // [wsplit, H, D] partial sums of dW_A
  char desc[512];
};

// Heads the score kernel covers per pass over X for model width D.
int score_heads_per_pass(int D);

namespace cat {
// Chunks per row of the multi-CTA softmax.
int softmax_parts(int N);
}

namespace cat {

// Fork points of the fast path's overlapped schedule: the chunk streams
// start after the spectrum of z*, after the score, or at once (their passes
// A need only V; passes B wait for the spectrum).
enum { FORK_SPECTRUM = 0, FORK_SCORE = 1, FORK_START = 2 };

// A range of batches and the stream its work goes to (default: all batches,
// the plan's stream).
struct Span {
  int b0 = 0;
  int nbat = -1;                 // -1: through the last batch
  cudaStream_t st = nullptr;
  bool own = false;              // true: use st instead of the plan's stream
  int nb(const cat_plan_s* p) const { return nbat < 0 ? p->B - b0 : nbat; }
  cudaStream_t stream(const cat_plan_s* p) const { return own ? st : p->stream; }
};

// Let `kernel` use all the dynamic shared memory the current device allows
// a block (its opt-in limit minus the kernel's static shared memory).  The
// limit is a property of the kernel, shared by every plan in the process,
// so it is always raised to the device maximum and never lowered to one
// plan's need.
template <typename K>
cudaError_t allow_max_smem(K kernel) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes a;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, kernel);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)a.sharedSizeBytes);
  return e;
}

// Launch `kernel` as the programmatic dependent of the kernel ahead of it
// on `st` (it may start before that one finishes; it calls pdl_wait before
// using that kernel's output).  Returns the launch's status.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // CAT_PDL=0: ordinary launches (the waits are then no-ops).
  if (const char* e = std::getenv("CAT_PDL")) cfg.numAttrs = e[0] == '0' ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launchers (enqueue on plan->stream).  Each returns cudaGetLastError().
cudaError_t launch_score(const cat_plan_s* p, const void* X, const void* WA,
                         const Span& sp = Span{});
// finish = false: only the chunk partials (the fast path's spectrum kernel
// applies the softmax itself).
cudaError_t launch_softmax(const cat_plan_s* p, const Span& sp = Span{}, bool finish = true);
cudaError_t launch_softmax_spectrum(const cat_plan_s* p);
cudaError_t launch_conv_smem(const cat_plan_s* p, const void* V, void* O);
// Register two-step circulant product for N = M² (M in {8, 14, 16, 32}).
cudaError_t setup_conv_reg(const cat_plan_s* p);
// conj: the product takes conj(FFT(z*)) (dV = circ(z*)^T dO of the backward).
cudaError_t launch_conv_reg(const cat_plan_s* p, const void* V, void* O, bool conj = false);
cudaError_t launch_softmax_spectrum_reg(const cat_plan_s* p);
// 2-D plan with reg2d: the scores a (channel-averaged 2-D correlation of Q
// and K) into z2 as (a, 0), and into out if given.
cudaError_t launch_scores2d_reg(const cat_plan_s* p, const void* Q, const void* K, float* out);
// Backward correlation dz*[b, h, k] = Σ_c Σ_i G[i, c] V[(i - k) mod N, c] into
// dzs by the register transform, for N = reg_m² on the shared-memory path.
cudaError_t launch_corr_reg(const cat_plan_s* p, const void* G, const void* V, float* dzs);
// At N = 32² (1-D) the correlation splits each row's pairs over 4 CTAs whose
// partial spectra (in the backward scratch, when it holds them) a finishing
// kernel adds, inverts and turns into dz* and dz (the softmax backward
// included): whether that fits, and the launch.
bool corr_reg_split_fits(const cat_plan_s* p);
cudaError_t launch_corr_reg_split(const cat_plan_s* p, const void* G, const void* V);
int conv_reg_pairs(int M);
size_t conv_reg_smem(int M, int P);
cudaError_t launch_fourstep_conv(const cat_plan_s* p, const void* V, void* O);
// Serialised fast-path circulant product; if ev is given, an event is
// recorded on the plan's stream after each pass (3 per chunk).
cudaError_t launch_fast_conv(const cat_plan_s* p, const void* V, void* O,
                             cudaEvent_t* ev = nullptr);
// Chunks of the fast path (launches of each of passes A, B, C per forward).
int fast_chunks(const cat_plan_s* p);
// Fast path pieces for the overlapped schedule: the spectrum of z* for
// (b, h) rows [row0, row0 + nrows), and passes A, B, C of one chunk of rows
// [bh0, bh0 + nb) with scratch buffer `slot`, all on stream st.  If
// before_b is given, pass B (the first to read the spectrum) waits for it.
// dep_a: the kernel ahead of this chunk's pass A on st is the previous
// chunk's pass C (pass A may then launch as its programmatic dependent).
// dependent: at N2 = 32 the spectrum kernel launches as the programmatic
// dependent of the kernel ahead (off for the stage-timed forward, whose
// events sit between them).  zs (N2 = 32 only): z* is written there too.
cudaError_t launch_fast_zspec(const cat_plan_s* p, int row0, int nrows, cudaStream_t st,
                              bool dependent = true, float* zs = nullptr);
cudaError_t launch_fast_chunk(const cat_plan_s* p, const void* V, void* O, int bh0, int nb,
                              int slot, cudaStream_t st, cudaEvent_t before_b = nullptr,
                              cudaEvent_t* after = nullptr, bool dep_a = false);

// Direct path (direct.cu): dynamic shared memory of a CTA, one-time
// attribute set-up, and the launch (fused: scores computed in the kernel;
// else from z2, which launch_score filled).
size_t direct_smem(int N, int D, int dh, int R, bool fused);
cudaError_t setup_direct_kernels(const cat_plan_s* p);
cudaError_t launch_direct(const cat_plan_s* p, const void* X, const void* WA, const void* V,
                          void* O, bool fused);

// 2-D plans on square grids of side 64, 96 or 128 (grid_pass.cu): whether
// the shape fits, the chunking and scratch size (no allocation), one-time
// attribute set-up, and the launch (V and O null: the scores only, into
// aout; else the forward, aout null).
bool grid_pass_supported(int h, int w, int dh);
int configure_grid_pass(cat_plan_s* p);
cudaError_t setup_grid_pass(const cat_plan_s* p);
cudaError_t launch_grid_pass(const cat_plan_s* p, const void* Q, const void* K, const void* V,
                             void* O, float* aout);

// Fused projection on the tensor cores (proj_tc.cu): V = X·W_V into V and
// the scores X·W_A into the plan's z2 in one pass over X (bf16, D % 64 == 0,
// H <= 16).  wt: project_workspace_bytes(D) of device memory for the
// transposed weights.
size_t project_workspace_bytes(int D);
cudaError_t setup_project_kernels();
cudaError_t launch_project(const cat_plan_s* p, const void* X, const void* WV, const void* WA,
                           void* V, void* wt);

// Shape validation and shared-memory-path configuration without allocation.
int validate(int B, int N, int D, int H, int dtype);
int configure_smem_path(cat_plan_s* p);

// One-time kernel attribute setup (dynamic shared memory limits).
cudaError_t setup_score_kernels(const cat_plan_s* p);
cudaError_t setup_smem_kernels(const cat_plan_s* p);
cudaError_t setup_fourstep_kernels(const cat_plan_s* p);
cudaError_t setup_fast_kernels(cat_plan_s* p);
size_t fast_tables_bytes(int N2);

// Backward pass (backward.cu).  launch_backward_dz: correlation passes and
// softmax backward into bw_dzs and bw_dz (needs z* in zs); with dV, also
// dV from the correlation's own transform of G (only where
// backward_dv_in_corr holds, with the spectrum of z* in zf, which its passes
// B take conjugated; the plan's stream joins the dV passes only at
// backward_join_dv).
// launch_backward_dense: dW_A and dX from bw_dz.  launch_reverse_scores:
// z2[n] <-> z2[(-n) mod N] in every row, so that the forward's spectrum and
// product kernels then give circ(z*)^T.
cudaError_t setup_backward_kernels(const cat_plan_s* p);
bool backward_dv_in_corr(const cat_plan_s* p);
// After a backward_dz with dV on the overlapped fast path: the plan's stream
// waits for the internal streams' last dV passes.
cudaError_t backward_join_dv(const cat_plan_s* p);
cudaError_t launch_backward_dz(const cat_plan_s* p, const void* G, const void* V,
                               void* dV = nullptr);
cudaError_t launch_backward_dense(const cat_plan_s* p, const void* X, const void* WA, void* dX,
                                  void* dWA);
cudaError_t launch_reverse_scores(const cat_plan_s* p);
int backward_wsplit(long long tokens, int D, int H, int sms);
// 2-D plan: the channel-averaged 2-D correlation of Q and K into the
// plan's scores z2 (ready for launch_softmax), and into out if given.
cudaError_t launch_scores2d(const cat_plan_s* p, const void* Q, const void* K,
                            float* out = nullptr);
// Fast path (head width 64, N = 512·N2): the correlation's pass A on dO
// (into s0, default scratch slot 0) and on V (s1, default slot 1), then its
// pass B into y[bhl][k2][n1] for rows [bh0, bh0 + nb), on stream st.
cudaError_t launch_fast_corr(const cat_plan_s* p, const void* G, const void* V, float2* y,
                             int bh0, int nb, cudaStream_t st, float2* s0 = nullptr,
                             float2* s1 = nullptr);
// Its pass C for N2 = 32: dz* rows [bh0, bh0 + nb) from y.
// Tensor-core dW_A and dX for bf16 data (dense_mma.cu): whether they serve
// this plan and these pointers, their one-time attribute set-up, the token
// splits of dW_A's partial sums (at most `most`), and the launches (dW_A's
// partial sums into part[nsplit][H][D], dX from the plan's dz).
bool dense_mma_ok(const cat_plan_s* p, const void* X, const void* dX);
cudaError_t setup_dense_mma();
int dwa_mma_splits(const cat_plan_s* p, int most);
cudaError_t launch_dwa_mma(const cat_plan_s* p, const void* X, float* part, int nsplit);
cudaError_t launch_dx_mma(const cat_plan_s* p, const void* WA, void* dX);

// Passes B and C (N2 = 32) on rows whose pass-A output already sits in
// scratch slot 0 (rows row_off .. row_off + nb - 1 of its tensor map, at
// scr), with the spectrum in p->zf, into O.
cudaError_t launch_fast_bc32(const cat_plan_s* p, float2* scr, void* O, int bh0, int nb,
                             int row_off, cudaStream_t st);
cudaError_t launch_fast_corr_c32(const cat_plan_s* p, const float2* y, float* dzs, int bh0,
                                 int nb, cudaStream_t st);

}  // namespace cat
