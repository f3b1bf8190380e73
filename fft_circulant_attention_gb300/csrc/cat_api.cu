// C ABI of libcat: plan construction, validation and the forward entry
// points declared in cat.h.  Host code only; the kernels live in score.cu,
// conv_smem.cu and fourstep.cu.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <vector>

#include "../../include/cat.h"
#include "cat_internal.h"

using cat::RadixPlan;

namespace {

constexpr int kSmemMaxN = 16384;             // longest single-CTA transform
constexpr size_t kConvSmemBudget = 64 << 10;  // preferred per-CTA tile (bytes)
constexpr size_t kFsSmemBudget = 100 << 10;
constexpr size_t kScratchBudget = 80ull << 20;  // live four-step scratch (L2-sized)
constexpr size_t kFastScratchBudget = 64ull << 20;
constexpr int kDirectMaxN = 1024;              // longest direct (O(N²)) product

bool seven_smooth(long n) {
  if (n < 1) return false;
  for (int p : {2, 3, 5, 7})
    while (n % p == 0) n /= p;
  return n == 1;
}

// Radices for a transform of length L (7-smooth): 8s, then a 4 or 2 for the
// rest of the power of two, then 7s, 5s, 3s.
bool make_radix_plan(int L, RadixPlan* rp) {
  std::memset(rp, 0, sizeof(*rp));
  rp->L = L;
  int n = L, k = 0;
  auto push = [&](int r) {
    if (k >= cat::kMaxPasses) return false;
    rp->radix[k++] = r;
    n /= r;
    return true;
  };
  while (n % 8 == 0)
    if (!push(8)) return false;
  if (n % 4 == 0 && !push(4)) return false;
  if (n % 2 == 0 && !push(2)) return false;
  for (int r : {7, 5, 3})
    while (n % r == 0)
      if (!push(r)) return false;
  if (n != 1) return false;
  rp->npass = k;
  return true;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Threads for `count` transforms of length L: about 16 values per thread,
// at least one warp, at most 1024.
int fft_threads(long count, int L) {
  long t = (count * L + 15) / 16;
  if (t < 32) t = 32;
  if (t > 1024) t = 1024;
  return round_up((int)t, 32);
}

// Pairs per CTA given a per-pair shared footprint, balanced across groups.
void split_pairs(int npair, int gmax, int* G, int* groups) {
  if (gmax < 1) gmax = 1;
  if (gmax > npair) gmax = npair;
  int g = (npair + gmax - 1) / gmax;
  *groups = g;
  *G = (npair + g - 1) / g;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? CAT_OK : CAT_ERR_CUDA; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

int check_shape(const cat_plan_s* p, int B, int N, int D, int H, int dtype) {
  if (B != p->B || N != p->N || D != p->D || H != p->H || dtype != p->dtype)
    return CAT_ERR_PLAN_MISMATCH;
  return CAT_OK;
}

int validate_shape(int B, int N, int D, int H, int dtype) {
  if (B < 0 || N < 1 || D < 1 || H < 1 || H > D) return CAT_ERR_INVALID_ARG;
  if (dtype != CAT_F32 && dtype != CAT_BF16) return CAT_ERR_INVALID_ARG;
  if (D > CAT_MAX_D || D % H != 0) return CAT_ERR_INVALID_ARG;
  if (N > CAT_MAX_N || !seven_smooth(N)) return CAT_ERR_UNSUPPORTED_N;
  // Largest element index must fit the kernels' size_t arithmetic; the
  // int-typed grid counts need B·H·N within 2^31.
  if ((long long)B * H * (long long)N > (1ll << 31)) return CAT_ERR_INVALID_ARG;
  return CAT_OK;
}

// Split N (> kSmemMaxN) into N1·N2, both 7-smooth and <= kSmemMaxN, with
// N1 >= N2 and N1 / N2 as small as possible.
bool split_fourstep(int N, int* N1, int* N2) {
  int best = -1;
  for (int a = 2; a <= kSmemMaxN && a < N; ++a) {
    if (N % a) continue;
    int b = N / a;
    if (b > kSmemMaxN || a < b || b < 2) continue;
    if (!seven_smooth(a) || !seven_smooth(b)) continue;
    if (best < 0 || a < best) best = a;
  }
  if (best < 0) return false;
  *N1 = best;
  *N2 = N / best;
  return true;
}

void free_events(cat_plan_s* p) {
  if (p->ev) {
    for (int i = 0; i < p->ev_per_call * p->timing_cap; ++i)
      if (p->ev[i]) cudaEventDestroy(p->ev[i]);
    delete[] p->ev;
  }
  p->ev = nullptr;
  p->timing_cap = p->timing_n = 0;
}

void free_plan(cat_plan_s* p) {
  if (!p) return;
  free_events(p);
  for (int k = 0; k < 2; ++k) {
    if (p->side[k]) cudaStreamDestroy(p->side[k]);
    if (p->ev_join[k]) cudaEventDestroy(p->ev_join[k]);
    if (p->ev_front[k]) cudaEventDestroy(p->ev_front[k]);
  }
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->gexec) cudaGraphExecDestroy(p->gexec);
  if (p->bgexec) cudaGraphExecDestroy(p->bgexec);
  if (p->cap) cudaStreamDestroy(p->cap);
  cudaFree(p->z2);
  cudaFree(p->zs);
  cudaFree(p->part);
  cudaFree(p->zf);
  cudaFree(p->tw);
  cudaFree(p->scratch);
  cudaFree(p->zscr);
  cudaFree(p->tabs);
  cudaFree(p->status);
  cudaFree(p->bw_scr);
  cudaFree(p->bw_dzs);
  cudaFree(p->bw_dz);
  cudaFree(p->bw_wpart);
  for (int k = 0; k < 2; ++k) {
    cudaFree(p->hx[k]);
    cudaFree(p->hv[k]);
    cudaFree(p->ho[k]);
    if (p->hsub[k]) free_plan(p->hsub[k]);
    if (p->hcp[k]) cudaStreamDestroy(p->hcp[k]);
    if (p->hev_in[k]) cudaEventDestroy(p->hev_in[k]);
    if (p->hev_done[k]) cudaEventDestroy(p->hev_done[k]);
    if (p->hev_out[k]) cudaEventDestroy(p->hev_out[k]);
  }
  cudaFree(p->hwa);
  cudaFree(p->pj_wt);
  delete p;
}

int score_launches(int H, int D) {
  int hpp = score_heads_per_pass(D);
  return (H + hpp - 1) / hpp;
}

int configure_fourstep(cat_plan_s* p, int N1, int N2);

// Whether the direct product can serve a shape: head width a multiple of 4
// (four columns a thread), at most 128, N <= kDirectMaxN, and a CTA of whole
// warps within 512 threads (dh/4 column threads times a row-group count
// that makes a multiple of 32).
bool direct_supported(const cat_plan_s* p) {
  if (p->dh % 4 != 0 || p->dh > 128 || p->N > kDirectMaxN) return false;
  const int ncg = p->dh / 4;
  int a = ncg, b = 32;
  while (b) { const int t = a % b; a = b; b = t; }
  return ncg * (32 / a) <= 512;
}

// Whether the direct product is the faster path for a supported shape.
// Measured on GB300 (forward, resident inputs): the register FFT kernels of
// the square lengths 8², 14², 16², 32² beat it (N = 196: 39 µs against
// 96 µs for B=64, D=384, H=6; N = 1024: 86 against 570 µs for GPT-2 small),
// while for other lengths up to 512 the block-FFT path is the slower one
// (N = 128: 92 against 35 µs for B=32, D=768, H=12 bf16; N = 512: 108
// against 90 µs for B=8).
constexpr int kDirectPreferMaxN = 512;
bool direct_preferred(const cat_plan_s* p) {
  const int N = p->N;
  for (int m : {8, 14, 16, 32})
    if (m * m == N) return false;
  return N <= kDirectPreferMaxN;
}

// Launch shape of the direct path (host only, no allocation).  TR, the rows
// a thread owns, is the largest of 8, 4, 2 that still gives a full wave of
// 256-thread CTAs.  A CTA covers as many rows as 512 threads allow (the
// whole row when it fits, so that the per-CTA softmax of the row is paid
// once); the row tile shrinks (down to 64-thread CTAs) until there are two
// CTAs per SM.  The scores are fused into the kernel when the row's X block
// is small enough that every CTA of the row may read it.
int configure_direct(cat_plan_s* p) {
  if (!direct_supported(p)) return CAT_ERR_UNSUPPORTED_N;
  p->path = cat::PATH_DIRECT;
  cat::DirectCfg& c = p->dir;
  const int N = p->N, ncg = p->dh / 4;
  const long bh = (long)p->B * p->H;
  const long sms = 152;
  c.TR = 2;
  for (int tr : {8, 4})
    if (bh * ((N + tr - 1) / tr) * ncg >= sms * 256) {
      c.TR = tr;
      break;
    }
  const int groups = (N + c.TR - 1) / c.TR;
  // Row groups per CTA: a multiple of `unit`, so that the CTA is a whole
  // number of warps (its block reductions shuffle over full warps).
  int g32 = ncg;
  for (int b2 = 32; b2;) { const int t = g32 % b2; g32 = b2; b2 = t; }
  const int unit = 32 / g32;
  auto ru = [&](int x) { return (x + unit - 1) / unit * unit; };
  const int nrg_cap = (512 / ncg) / unit * unit;
  int nrg = ru(groups) < nrg_cap ? ru(groups) : nrg_cap;
  const int nrg_min = ru((64 + ncg - 1) / ncg);
  auto ctas = [&](int g) { return bh * ((N + c.TR * g - 1) / (c.TR * g)); };
  for (;;) {
    const int nx = ru(nrg / 2);
    if (nx >= nrg || nx < nrg_min || ctas(nrg) >= 2 * sms) break;
    nrg = nx;
  }
  c.nrg = nrg;
  c.R = c.TR * nrg;
  c.threads = ncg * nrg;
  const size_t es = p->dtype == CAT_BF16 ? 2 : 4;
  const double fused_bytes = (double)ctas(nrg) * N * p->D * es;
  c.fused = (long)N * p->D <= (1L << 17) && fused_bytes <= 64e6;
  if (const char* f = std::getenv("CAT_DIRECT_FUSED")) c.fused = std::strcmp(f, "0") != 0;
  c.smem = cat::direct_smem(N, p->D, p->dh, c.R, c.fused != 0);
  p->launches = c.fused ? 1 : score_launches(p->H, p->D) + 1;
  return CAT_OK;
}

int choose_path(cat_plan_s* p) {
  const int N = p->N;
  // CAT_FORCE_PATH=fourstep sends short sequences down the multi-pass path
  // too (debugging and testing of that path at small sizes); =direct takes
  // the direct product wherever it is supported; =smem never takes it.
  const char* force = std::getenv("CAT_FORCE_PATH");
  if (direct_supported(p) &&
      (force ? std::strcmp(force, "direct") == 0 : direct_preferred(p)))
    return configure_direct(p);
  int n1 = 0, n2 = 0;
  const bool force_fs = force && std::strcmp(force, "fourstep") == 0 && split_fourstep(N, &n1, &n2);
  const bool allow_fast = !(force && (std::strcmp(force, "fourstep") == 0 ||
                                      std::strcmp(force, "smem") == 0));
  // Fast three-pass path: head width 64 and N = 512·N2, N2 in {32..256}.
  if (allow_fast && p->dh == 64 && N % 512 == 0) {
    const int N2 = N / 512;
    if (N2 == 32 || N2 == 64 || N2 == 128 || N2 == 256) {
      p->path = cat::PATH_FAST;
      cat::FourStepCfg& f = p->fs;
      f.N1 = 512;
      f.N2 = N2;
      if (!make_radix_plan(f.N1, &f.rp1) || !make_radix_plan(N2, &f.rp2) ||
          !make_radix_plan(N, &p->rpN))
        return CAT_ERR_UNSUPPORTED_N;
      f.G = 32;
      f.groups = 1;
      f.P = 32;
      // Chunks of (b, h) rows stay inside one batch; two scratch slots let
      // two chunks be in flight on the plan's two internal streams.  A slot
      // takes half the scratch budget: 8 heads at N = 16384 (one batch of
      // 16 heads runs in 68 µs with chunks of 8, 127 µs with single heads),
      // one head at N = 131072.
      const size_t per_bh = (size_t)N * 32 * sizeof(float2);
      long chunk = (long)(kFastScratchBudget / 2 / per_bh);
      if (const char* env = std::getenv("CAT_CHUNK_BH")) chunk = std::atol(env);
      if (chunk < 1) chunk = 1;
      if (chunk > p->H) chunk = p->H;
      f.chunk_bh = (int)chunk;
      p->scratch_bytes = 2 * (size_t)f.chunk_bh * per_bh;
      const int chunks_per_batch = (int)((p->H + chunk - 1) / chunk);
      // Front once — the score passes, then the spectrum of z* (one launch for
      // N2 = 32; softmax partials and two launches for longer rows) — then
      // passes A, B, C per chunk.
      p->launches = score_launches(p->H, p->D) + (f.N2 == 32 ? 1 : 3) + 3 * p->B * chunks_per_batch;
      return CAT_OK;
    }
  }
  if (N <= kSmemMaxN && !force_fs) return cat::configure_smem_path(p);
  if (!split_fourstep(N, &n1, &n2)) return CAT_ERR_UNSUPPORTED_N;
  return configure_fourstep(p, n1, n2);
}

// The generic four-step path for the split N = N1·N2 (both 7-smooth, at
// most 16384; a 2-D plan passes N1 = w, N2 = h).
int configure_fourstep(cat_plan_s* p, int N1, int N2) {
  const int N = p->N;
  p->path = cat::PATH_FOURSTEP;
  cat::FourStepCfg& f = p->fs;
  f.N1 = N1;
  f.N2 = N2;
  if (!make_radix_plan(f.N1, &f.rp1) || !make_radix_plan(f.N2, &f.rp2))
    return CAT_ERR_UNSUPPORTED_N;
  if (!make_radix_plan(N, &p->rpN)) return CAT_ERR_UNSUPPORTED_N;
  const size_t c8 = sizeof(float2);
  // Pairs per CTA: pass B holds TB·(G+1) signals of length N1.
  int gmax = (int)(kFsSmemBudget / ((size_t)f.N1 * c8)) - 1;
  if (gmax > 16) gmax = 16;
  split_pairs(p->npair, gmax, &f.G, &f.groups);
  f.P = p->npair + 1;
  // Tiles: as many n1 (k2) slots as fit the budget, dividing N1 (N2).
  f.TA = 1;
  for (int t = 2; t <= 64; ++t)
    if (f.N1 % t == 0 && (size_t)t * (f.G + 1) * f.N2 * c8 <= kFsSmemBudget) f.TA = t;
  f.TB = 1;
  for (int t = 2; t <= 64; ++t)
    if (f.N2 % t == 0 && (size_t)t * (f.G + 1) * f.N1 * c8 <= kFsSmemBudget) f.TB = t;
  f.smemA = (size_t)f.TA * (f.G + 1) * f.N2 * c8;
  f.smemB = (size_t)f.TB * (f.G + 1) * f.N1 * c8;
  f.smemC = (size_t)f.TA * f.G * f.N2 * c8;
  f.threadsA = fft_threads((long)f.TA * (f.G + 1), f.N2);
  f.threadsB = fft_threads((long)f.TB * (f.G + 1), f.N1);
  f.threadsC = fft_threads((long)f.TA * f.G, f.N2);
  if ((long)f.TA * (f.G + 1) * f.N2 > (long)cat::vals_capacity(f.rp2) * f.threadsA ||
      (long)f.TB * (f.G + 1) * f.N1 > (long)cat::vals_capacity(f.rp1) * f.threadsB ||
      (long)f.TA * f.G * f.N2 > (long)cat::vals_capacity(f.rp2) * f.threadsC)
    return CAT_ERR_UNSUPPORTED_N;
  size_t per_bh = (size_t)N * f.P * c8;
  long chunk = (long)(kScratchBudget / per_bh);
  if (const char* env = std::getenv("CAT_CHUNK_BH")) chunk = std::atol(env);
  if (chunk < 1) chunk = 1;
  long rows = (long)p->B * p->H;
  if (chunk > rows) chunk = rows > 0 ? rows : 1;
  f.chunk_bh = (int)chunk;
  p->scratch_bytes = (size_t)f.chunk_bh * per_bh;
  p->launches = score_launches(p->H, p->D) + 2 + 3 * (int)((rows + chunk - 1) / chunk);
  return CAT_OK;
}

void describe(cat_plan_s* p) {
  char rad[128] = {0};
  auto radstr = [](const RadixPlan& rp, char* out, size_t len) {
    size_t o = 0;
    for (int i = 0; i < rp.npass && o + 4 < len; ++i)
      o += (size_t)std::snprintf(out + o, len - o, i ? "x%d" : "%d", rp.radix[i]);
  };
  if (p->path == cat::PATH_DIRECT) {
    std::snprintf(p->desc, sizeof(p->desc),
                  "path=direct N=%d TR=%d R=%d threads=%d fused=%d smem=%zu workspace=%zu "
                  "launches=%d",
                  p->N, p->dir.TR, p->dir.R, p->dir.threads, p->dir.fused, p->dir.smem,
                  p->workspace_bytes, p->launches);
  } else if (p->path == cat::PATH_SMEM) {
    radstr(p->rpN, rad, sizeof(rad));
    std::snprintf(p->desc, sizeof(p->desc),
                  "path=smem N=%d radices=%s reg_m=%d G=%d groups=%d threads=%d smem=%zu "
                  "spec_threads=%d workspace=%zu launches=%d",
                  p->N, rad, p->sm.reg_m, p->sm.G, p->sm.groups, p->sm.threads, p->sm.smem,
                  p->sm.spec_threads, p->workspace_bytes, p->launches);
  } else if (p->path == cat::PATH_FAST) {
    std::snprintf(p->desc, sizeof(p->desc),
                  "path=fast N=%d N1=%d N2=%d chunk_bh=%d scratch=%zu workspace=%zu graph=%d "
                  "launches=%d",
                  p->N, p->fs.N1, p->fs.N2, p->fs.chunk_bh, p->scratch_bytes,
                  p->workspace_bytes, p->use_graph, p->launches);
  } else if (p->gp2d) {
    std::snprintf(p->desc, sizeof(p->desc),
                  "path=grid2d gp=1 N=%d M=%d(32x%d) chunk_bh=%d scratch=%zu workspace=%zu "
                  "launches=%d",
                  p->N, p->gp.M, p->gp.R, p->gp.chunk, p->scratch_bytes, p->workspace_bytes,
                  p->launches);
  } else {
    char r1[64] = {0}, r2[64] = {0};
    radstr(p->fs.rp1, r1, sizeof(r1));
    radstr(p->fs.rp2, r2, sizeof(r2));
    std::snprintf(p->desc, sizeof(p->desc),
                  "path=%s%s N=%d N1=%d(%s) N2=%d(%s) G=%d groups=%d TA=%d TB=%d "
                  "threads=%d/%d/%d smem=%zu/%zu/%zu chunk_bh=%d scratch=%zu workspace=%zu "
                  "launches=%d",
                  p->twod ? "grid2d" : "fourstep", p->reg2d ? " reg2d=1" : "", p->N,
                  p->fs.N1, r1, p->fs.N2, r2, p->fs.G,
                  p->fs.groups, p->fs.TA, p->fs.TB,
                  p->fs.threadsA, p->fs.threadsB, p->fs.threadsC, p->fs.smemA, p->fs.smemB,
                  p->fs.smemC, p->fs.chunk_bh, p->scratch_bytes, p->workspace_bytes,
                  p->launches);
  }
}

// Score, softmax and (shared-memory path) spectrum of z* into the plan.
int run_front(cat_plan_s* p, const void* X, const void* WA) {
  cudaError_t e = cat::launch_score(p, X, WA);
  if (e != cudaSuccess) return CAT_ERR_CUDA;
  if (p->path == cat::PATH_SMEM)
    e = cat::launch_softmax_spectrum(p);
  else
    e = cat::launch_softmax(p);
  return map_cuda(e);
}


// Device workspace a configured plan allocates at creation: scores (fp32
// pairs) and z*, the twiddle table, the spectrum of z* (shared-memory and
// fast paths), the fast path's first-pass spectrum and tables, and the
// multi-pass scratch.
size_t planned_workspace(const cat_plan_s* p) {
  const size_t rowsN = (size_t)p->B * p->H * p->N;
  const bool fast = p->path == cat::PATH_FAST;
  return rowsN * (sizeof(float) + sizeof(float2)) + (size_t)p->N * sizeof(float2) +
         ((p->path == cat::PATH_SMEM || fast || p->reg2d) ? rowsN * sizeof(float2) : 0) +
         (fast ? rowsN * sizeof(float2) : 0) +
         (p->path != cat::PATH_SMEM ? p->scratch_bytes : 0) +
         (fast ? cat::fast_tables_bytes(p->fs.N2) : 0);
}

int configure_corr(cat_plan_s* p, int N1, int N2);

// Launch shapes of the backward correlation (host only, no allocation).
// Rows up to 4096 are transformed whole in pass B (N1 = N, N2 = 1); longer
// ones use the four-step split of the long-sequence forward path.
int configure_backward(cat_plan_s* p) {
  cat::BwCfg& w = p->bw;
  std::memset(&w, 0, sizeof(w));
  const int N = p->N;
  const size_t c8 = sizeof(float2);
  if (p->path == cat::PATH_FAST) {
    // The fast path's pass A and the register kernel fsf_corr_b (both in
    // its scratch slots and chunks), then pass C on one signal per row.
    w.fast = 1;
    w.N1 = p->fs.N1;
    w.N2 = p->fs.N2;
    w.rp1 = p->fs.rp1;
    w.rp2 = p->fs.rp2;
    w.Q = 1;
    w.TC = 1;
    for (int t = 2; t <= 64; ++t)
      if (w.N1 % t == 0 && (size_t)t * w.N2 * c8 <= kFsSmemBudget) w.TC = t;
    w.smemC = (size_t)w.TC * w.N2 * c8;
    w.threadsC = fft_threads(w.TC, w.N2);
    if ((long)w.TC * w.N2 > (long)cat::vals_capacity(w.rp2) * w.threadsC)
      return CAT_ERR_UNSUPPORTED_N;
    w.chunk_bh = p->fs.chunk_bh;
    // y, the correlation's one signal per row: every row's at N2 = 32 (the
    // overlapped chunks leave theirs for one pass-C launch at the end), a
    // chunk's otherwise.
    const size_t yrows = w.N2 == 32 ? (size_t)p->B * p->H : (size_t)w.chunk_bh;
    w.scratch_bytes = yrows * N * c8;
    w.wsplit = cat::backward_wsplit((long long)p->B * N, p->D, p->H, p->sms > 0 ? p->sms : 148);
    return CAT_OK;
  }
  int n1 = N, n2 = 1;
  if (p->twod) {
    n1 = p->grid_w;
    n2 = p->grid_h;
  } else if (N > 4096 && !split_fourstep(N, &n1, &n2)) {
    return CAT_ERR_UNSUPPORTED_N;
  }
  return configure_corr(p, n1, n2);
}

// Launch shapes of the generic correlation passes for the split N = N1·N2.
int configure_corr(cat_plan_s* p, int N1, int N2) {
  cat::BwCfg& w = p->bw;
  const int N = p->N;
  const size_t c8 = sizeof(float2);
  w.N1 = N1;
  w.N2 = N2;
  if (!make_radix_plan(w.N1, &w.rp1) || !make_radix_plan(w.N2, &w.rp2))
    return CAT_ERR_UNSUPPORTED_N;
  const int np = p->npair;
  w.Q = 2 * np;
  // Pass A: up to 16 pairs (32 signals) per CTA, then as many n1 as fit.
  int gmax = (int)(kFsSmemBudget / (2 * (size_t)w.N2 * c8));
  if (gmax > 16) gmax = 16;
  if (gmax < 1) return CAT_ERR_UNSUPPORTED_N;
  split_pairs(np, gmax, &w.GA, &w.groupsA);
  w.TA = 1;
  for (int t = 2; t <= 64; ++t)
    if (w.N1 % t == 0 && (size_t)t * 2 * w.GA * w.N2 * c8 <= kFsSmemBudget) w.TA = t;
  w.smemA = (size_t)w.TA * 2 * w.GA * w.N2 * c8;
  w.threadsA = fft_threads((long)w.TA * 2 * w.GA, w.N2);
  // Pass B: chunks of up to 8 pairs plus the accumulator, TB k2 per CTA.
  w.GB = np < 8 ? np : 8;
  w.TB = 0;
  for (; w.GB >= 1 && !w.TB; --w.GB) {
    for (int t = 1; t <= 64; ++t)
      if (w.N2 % t == 0 && (size_t)t * (2 * w.GB + 1) * w.N1 * c8 <= kFsSmemBudget) w.TB = t;
    if (w.TB) break;
  }
  if (w.GB < 1 || !w.TB) return CAT_ERR_UNSUPPORTED_N;
  w.smemB = (size_t)w.TB * (2 * w.GB + 1) * w.N1 * c8;
  w.threadsB = fft_threads((long)w.TB * 2 * w.GB, w.N1);
  // Pass C: one signal per n1, TC n1 per CTA.
  w.TC = 1;
  for (int t = 2; t <= 64; ++t)
    if (w.N1 % t == 0 && (size_t)t * w.N2 * c8 <= kFsSmemBudget) w.TC = t;
  w.smemC = (size_t)w.TC * w.N2 * c8;
  w.threadsC = fft_threads(w.TC, w.N2);
  if ((long)w.TA * 2 * w.GA * w.N2 > (long)cat::vals_capacity(w.rp2) * w.threadsA ||
      (long)w.TB * 2 * w.GB * w.N1 > (long)cat::vals_capacity(w.rp1) * w.threadsB ||
      (long)w.TB * w.N1 > (long)cat::vals_capacity(w.rp1) * w.threadsB ||
      (long)w.TC * w.N2 > (long)cat::vals_capacity(w.rp2) * w.threadsC)
    return CAT_ERR_UNSUPPORTED_N;
  const size_t per_bh = (size_t)N * w.Q * c8;
  long chunk = (long)(kScratchBudget / per_bh);
  if (chunk < 1) chunk = 1;
  const long rows = (long)p->B * p->H;
  if (chunk > rows) chunk = rows > 0 ? rows : 1;
  w.chunk_bh = (int)chunk;
  w.scratch_bytes = (size_t)w.chunk_bh * per_bh;
  w.wsplit = cat::backward_wsplit((long long)p->B * N, p->D, p->H, p->sms > 0 ? p->sms : 148);
  return CAT_OK;
}

// Configure and allocate the backward workspace at the first backward call.
int ensure_backward(cat_plan_s* p) {
  if (p->bw_ready) return CAT_OK;
  int st = configure_backward(p);
  if (st != CAT_OK) return st;
  const size_t rowsN = (size_t)p->B * p->H * p->N;
  auto alloc = [&](void** ptr, size_t bytes) {
    if (bytes == 0) bytes = 16;
    return cudaMalloc(ptr, bytes) == cudaSuccess;
  };
  bool ok = alloc((void**)&p->bw_scr, p->bw.scratch_bytes) &&
            alloc((void**)&p->bw_dzs, rowsN * sizeof(float)) &&
            alloc((void**)&p->bw_dz, rowsN * sizeof(float)) &&
            alloc((void**)&p->bw_wpart, (size_t)p->bw.wsplit * p->H * p->D * sizeof(float));
  if (!ok) {
    cudaGetLastError();
    cudaFree(p->bw_scr); cudaFree(p->bw_dzs); cudaFree(p->bw_dz); cudaFree(p->bw_wpart);
    p->bw_scr = nullptr; p->bw_dzs = p->bw_dz = p->bw_wpart = nullptr;
    return CAT_ERR_ALLOC;
  }
  if (cat::setup_backward_kernels(p) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p->bw_scr); cudaFree(p->bw_dzs); cudaFree(p->bw_dz); cudaFree(p->bw_wpart);
    p->bw_scr = nullptr; p->bw_dzs = p->bw_dz = p->bw_wpart = nullptr;
    return CAT_ERR_CUDA;
  }
  p->bw_ready = 1;
  return CAT_OK;
}

// Score and softmax into the plan (z* in zs on every path), then the
// correlation and the softmax backward (dz* and dz in the plan).
int run_backward_front(cat_plan_s* p, const void* X, const void* WA, const void* V,
                       const void* G) {
  cudaError_t e = cat::launch_score(p, X, WA);
  if (e == cudaSuccess) e = cat::launch_softmax(p);
  if (e == cudaSuccess) e = cat::launch_backward_dz(p, G, V);
  return map_cuda(e);
}
}  // namespace

namespace cat {

// Launch configuration of the shared-memory path for an already-validated
// shape (N <= 16384), without touching the device or allocating: fills the
// radix plan, the SmemCfg and the launch count of *p.
int configure_smem_path(cat_plan_s* p) {
  const int N = p->N;
  if (N > kSmemMaxN) return CAT_ERR_UNSUPPORTED_N;
  p->path = cat::PATH_SMEM;
  if (!make_radix_plan(N, &p->rpN)) return CAT_ERR_UNSUPPORTED_N;
  cat::SmemCfg& s = p->sm;
  size_t per = (size_t)N * sizeof(float2);
  split_pairs(p->npair, (int)(kConvSmemBudget / per), &s.G, &s.groups);
  s.tstride = N;
  s.smem = (size_t)s.G * s.tstride * sizeof(float2);
  s.threads = fft_threads(s.G, N);
  s.spec_threads = fft_threads(1, N);
  s.spec_smem = per;
  if ((long)s.G * N > (long)cat::vals_capacity(p->rpN) * s.threads) return CAT_ERR_UNSUPPORTED_N;
  if ((long)N > (long)cat::vals_capacity(p->rpN) * s.spec_threads) return CAT_ERR_UNSUPPORTED_N;
  // Square lengths with a register transform of the side take the two-step
  // register kernel for the circulant product (CAT_SMEM_REG=0: block FFT).
  s.reg_m = 0;
  const char* env = std::getenv("CAT_SMEM_REG");
  if (!(env && std::strcmp(env, "0") == 0)) {
    for (int m : {8, 14, 16, 32})
      if (m * m == N) s.reg_m = m;
  }
  if (s.reg_m) {
    s.G = cat::conv_reg_pairs(s.reg_m);
    s.groups = (p->npair + s.G - 1) / s.G;
    s.smem = cat::conv_reg_smem(s.reg_m, s.G);
    s.threads = s.reg_m * s.G;
  }
  p->launches = score_launches(p->H, p->D) + 2;
  return CAT_OK;
}

// Shape validation shared with the plan constructor.
int validate(int B, int N, int D, int H, int dtype) { return validate_shape(B, N, D, H, dtype); }

}  // namespace cat

extern "C" {

namespace {

// Fast path, overlapped schedule: the score and the spectrum of z* (each a
// single launch over all batches) on the plan's stream; the chunks' passes
// alternate between the two internal streams, one scratch slot each.  The
// internal streams fork from the plan's stream at p->fork_at; when that is
// before the spectrum, each waits for it just before its first pass B, so
// the first passes A run beside the score and the spectrum.  Both join back
// into the plan's stream at the end.
// `between`, if given, enqueues further work on the plan's stream after the
// spectrum and the chunks are enqueued and before the join, so that it runs
// beside the chunks (the backward's dense gradients beside its dV).
cudaError_t run_fast_overlapped(cat_plan_s* p, const void* X, const void* WA, const void* V,
                                void* O, bool score = true,
                                const std::function<cudaError_t()>* between = nullptr) {
  cudaError_t e = cudaSuccess;
  auto fork = [&]() {
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_fork, p->stream);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k)
      e = cudaStreamWaitEvent(p->side[k], p->ev_fork, 0);
  };
  if (p->fork_at == cat::FORK_START) fork();
  if (e == cudaSuccess && score) e = cat::launch_score(p, X, WA);
  if (p->fork_at == cat::FORK_SCORE) fork();
  if (e == cudaSuccess) e = cat::launch_fast_zspec(p, 0, p->B * p->H, p->stream);
  if (p->fork_at == cat::FORK_SPECTRUM) fork();
  else if (e == cudaSuccess) e = cudaEventRecord(p->ev_front[0], p->stream);
  bool waited[2] = {p->fork_at == cat::FORK_SPECTRUM, p->fork_at == cat::FORK_SPECTRUM};
  int g = 0;
  for (int b = 0; b < p->B && e == cudaSuccess; ++b)
    for (int h0 = 0; h0 < p->H && e == cudaSuccess; h0 += p->fs.chunk_bh, ++g) {
      const int nb = p->H - h0 < p->fs.chunk_bh ? p->H - h0 : p->fs.chunk_bh;
      const int k = g & 1;
      e = cat::launch_fast_chunk(p, V, O, b * p->H + h0, nb, k, p->side[k],
                                 waited[k] ? nullptr : p->ev_front[0], nullptr, g >= 2);
      waited[k] = true;
    }
  if (e == cudaSuccess && between) e = (*between)();
  for (int k = 0; k < 2; ++k) {
    cudaError_t e2 = cudaEventRecord(p->ev_join[k], p->side[k]);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(p->stream, p->ev_join[k], 0);
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

// The forward's schedule without stage events: the fast path's overlapped
// schedule, else the score, the softmax (with the spectrum of z* on the
// shared-memory path) and the circulant product, or the direct product.
cudaError_t forward_schedule(cat_plan_s* p, const void* X, const void* WA, const void* V,
                             void* O) {
  if (p->path == cat::PATH_FAST) return run_fast_overlapped(p, X, WA, V, O);
  if (p->path == cat::PATH_DIRECT) {
    cudaError_t e = p->dir.fused ? cudaSuccess : cat::launch_score(p, X, WA);
    if (e == cudaSuccess) e = cat::launch_direct(p, X, WA, V, O, p->dir.fused != 0);
    return e;
  }
  cudaError_t e = cat::launch_score(p, X, WA);
  if (e == cudaSuccess)
    e = p->path == cat::PATH_SMEM ? cat::launch_softmax_spectrum(p) : cat::launch_softmax(p);
  if (e == cudaSuccess)
    e = p->path == cat::PATH_SMEM ? cat::launch_conv_smem(p, V, O)
                                  : cat::launch_fourstep_conv(p, V, O);
  return e;
}

// The forward through a CUDA graph: the schedule is captured on the private
// stream (on the fast path its fork and join events pull the two internal
// streams into the capture), instantiated once, updated in place when the
// call's pointers change, and launched on the plan's stream.  A graph launch
// replaces the schedule's separate launches and event operations.
cudaError_t launch_forward_graph(cat_plan_s* p, const void* X, const void* WA, const void* V,
                              void* O) {
  if (!p->gexec || X != p->gX || WA != p->gWA || V != p->gV || O != p->gO) {
    cudaStream_t saved = p->stream;
    p->stream = p->cap;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      const cudaError_t e1 = forward_schedule(p, X, WA, V, O);
      const cudaError_t e2 = cudaStreamEndCapture(p->cap, &g);
      e = e1 != cudaSuccess ? e1 : e2;
    }
    p->stream = saved;
    if (e == cudaSuccess && p->gexec) {
      cudaGraphExecUpdateResultInfo info;
      if (cudaGraphExecUpdate(p->gexec, g, &info) != cudaSuccess) {
        cudaGetLastError();
        cudaGraphExecDestroy(p->gexec);
        p->gexec = nullptr;
      }
    }
    if (e == cudaSuccess && !p->gexec) e = cudaGraphInstantiate(&p->gexec, g, 0);
    if (g) cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      if (p->gexec) cudaGraphExecDestroy(p->gexec);
      p->gexec = nullptr;
      return e;
    }
    p->gX = X; p->gWA = WA; p->gV = V; p->gO = O;
  }
  return cudaGraphLaunch(p->gexec, p->stream);
}

}  // namespace

namespace {
int create_plan(cat_plan_t* out, int B, int N, int D, int H, int dtype, void* stream, int gh,
                int gw);
}

int cat_plan_create(cat_plan_t* out, int B, int N, int D, int H, int dtype, void* stream) {
  return create_plan(out, B, N, D, H, dtype, stream, 0, 0);
}

int cat_plan_create_2d(cat_plan_t* out, int B, int h, int w, int D, int H, int dtype,
                       void* stream) {
  if (!out) return CAT_ERR_INVALID_ARG;
  *out = nullptr;
  if (h < 1 || w < 1) return CAT_ERR_INVALID_ARG;
  if (h > kSmemMaxN || w > kSmemMaxN || !seven_smooth(h) || !seven_smooth(w))
    return CAT_ERR_UNSUPPORTED_N;
  if ((long long)h * w > CAT_MAX_N) return CAT_ERR_UNSUPPORTED_N;
  return create_plan(out, B, h * w, D, H, dtype, stream, h, w);
}

namespace {
int create_plan(cat_plan_t* out, int B, int N, int D, int H, int dtype, void* stream, int gh,
                int gw) {
  if (!out) return CAT_ERR_INVALID_ARG;
  *out = nullptr;
  int st = validate_shape(B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  cat_plan_s* p = new (std::nothrow) cat_plan_s();
  if (!p) return CAT_ERR_ALLOC;
  p->B = B; p->N = N; p->D = D; p->H = H; p->dtype = dtype;
  p->dh = D / H;
  p->npair = (p->dh + 1) / 2;
  p->stream = (cudaStream_t)stream;
  if (gh > 0) {
    // 2-D plan: the generic four-step passes over the grid (N1 = w, N2 = h)
    // without twiddles; the scores come from the correlation passes.
    p->twod = 1;
    p->grid_h = gh;
    p->grid_w = gw;
    st = configure_fourstep(p, gw, gh);
    // Square grids of a register-DFT side take the register kernels
    // (CAT_2D_REG=0: the generic passes).
    const char* r2 = std::getenv("CAT_2D_REG");
    if (st == CAT_OK && gh == gw && (gh == 8 || gh == 14 || gh == 16 || gh == 32) &&
        !(r2 && std::strcmp(r2, "0") == 0)) {
      p->reg2d = 1;
      cat::SmemCfg& sc = p->sm;
      sc.reg_m = gh;
      sc.G = cat::conv_reg_pairs(gh);
      sc.groups = (p->npair + sc.G - 1) / sc.G;
      sc.smem = cat::conv_reg_smem(gh, sc.G);
      sc.threads = gh * sc.G;
      p->launches = 3;
    } else if (st == CAT_OK && cat::grid_pass_supported(gh, gw, p->dh) &&
               !(r2 && std::strcmp(r2, "0") == 0)) {
      // Square grids of side 64, 96 or 128: the row/column passes.
      p->gp2d = 1;
      st = cat::configure_grid_pass(p);
      p->scratch_bytes = p->gp.scratch_bytes;
      const int rows = B * H;
      p->launches = 5 * ((rows + p->gp.chunk - 1) / p->gp.chunk);
    }
  } else {
    st = choose_path(p);
  }
  if (st != CAT_OK) { delete p; return st; }
  // Default fork point: after the score when the spectrum is one launch
  // (N2 = 32, where the first passes A then overlap it), else after it.
  p->fork_at = p->path == cat::PATH_FAST && p->fs.N2 == 32 ? cat::FORK_SCORE : cat::FORK_SPECTRUM;
  if (const char* sc = std::getenv("CAT_FORK"))
    p->fork_at = std::strcmp(sc, "start") == 0   ? cat::FORK_START
                 : std::strcmp(sc, "score") == 0 ? cat::FORK_SCORE
                                                 : cat::FORK_SPECTRUM;
  // Fast-path passes as programmatic dependents of the pass ahead
  // (CAT_PDL_FAST=0 off, "end": signal at each CTA's end, else at its start).
  p->fast_pdl = 2;
  if (const char* sc = std::getenv("CAT_PDL_FAST"))
    p->fast_pdl = std::strcmp(sc, "0") == 0 ? 0 : std::strcmp(sc, "end") == 0 ? 1 : 2;
  if (const char* sc = std::getenv("CAT_SCORE")) {
    p->score_cuda_cores = std::strcmp(sc, "cuda") == 0;
    p->score_path = std::strcmp(sc, "mma") == 0 ? 1 : 0;
  }

  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return CAT_ERR_CUDA;
  }
  const size_t rowsN = (size_t)B * H * N;
  auto alloc = [&](void** ptr, size_t bytes) {
    if (bytes == 0) bytes = 16;
    return cudaMalloc(ptr, bytes) == cudaSuccess;
  };
  bool ok = alloc((void**)&p->z2, rowsN * sizeof(float2)) &&
            alloc((void**)&p->zs, rowsN * sizeof(float)) &&
            alloc((void**)&p->part, (size_t)B * H * cat::softmax_parts(N) * sizeof(float2)) &&
            alloc((void**)&p->tw, (size_t)N * sizeof(float2)) &&
            alloc((void**)&p->status, sizeof(unsigned int));
  if (ok && (p->path == cat::PATH_SMEM || p->path == cat::PATH_FAST || p->reg2d))
    ok = alloc((void**)&p->zf, rowsN * sizeof(float2));
  if (ok && p->path == cat::PATH_FAST) ok = alloc((void**)&p->zscr, rowsN * sizeof(float2));
  if (ok && p->path == cat::PATH_FAST)
    ok = alloc((void**)&p->tabs, cat::fast_tables_bytes(p->fs.N2));
  if (ok && p->path != cat::PATH_SMEM) ok = alloc((void**)&p->scratch, p->scratch_bytes);
  if (!ok) { cudaGetLastError(); free_plan(p); return CAT_ERR_ALLOC; }
  p->workspace_bytes = planned_workspace(p);

  // Twiddle table exp(-2πi j/N), evaluated in fp64 and rounded once.
  std::vector<float2> tw((size_t)N);
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = 0; j < N; ++j) {
    double a = -two_pi * (double)j / (double)N;
    tw[j] = make_float2((float)std::cos(a), (float)std::sin(a));
  }
  cudaError_t e = cudaMemcpy(p->tw, tw.data(), (size_t)N * sizeof(float2), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p->status, 0, sizeof(unsigned int));
  if (e == cudaSuccess) e = cat::setup_score_kernels(p);
  if (e == cudaSuccess)
    e = p->path == cat::PATH_SMEM       ? cat::setup_smem_kernels(p)
        : p->path == cat::PATH_FOURSTEP ? cat::setup_fourstep_kernels(p)
        : p->path == cat::PATH_DIRECT   ? cat::setup_direct_kernels(p)
                                        : cat::setup_fast_kernels(p);
  if (e == cudaSuccess && p->reg2d) e = cat::setup_conv_reg(p);
  if (e == cudaSuccess && p->gp2d) e = cat::setup_grid_pass(p);
  if (e == cudaSuccess && p->path == cat::PATH_FAST) {
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
      e = cudaStreamCreateWithFlags(&p->side[k], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_join[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_front[k], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming);
  }
  // Graph replay (CAT_GRAPH=0: direct launches) of every 1-D plan's forward
  // and backward, captured on a private stream.
  if (e == cudaSuccess && !p->twod) {
    p->use_graph = 1;
    if (const char* g = std::getenv("CAT_GRAPH")) p->use_graph = std::strcmp(g, "0") != 0;
    if (p->use_graph) e = cudaStreamCreateWithFlags(&p->cap, cudaStreamNonBlocking);
  }
  if (e != cudaSuccess) { free_plan(p); return CAT_ERR_CUDA; }
  if (p->twod) {
    st = ensure_backward(p);
    if (st != CAT_OK) { free_plan(p); return st; }
  }
  describe(p);
  if (std::getenv("CAT_LOG")) std::fprintf(stderr, "[cat] %s\n", p->desc);
  *out = p;
  return CAT_OK;
}
}  // namespace

int cat_plan_query(int B, int N, int D, int H, int dtype, size_t* workspace_bytes, char* desc,
                   int len) {
  int st = validate_shape(B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  cat_plan_s q{};
  q.B = B; q.N = N; q.D = D; q.H = H; q.dtype = dtype;
  q.dh = D / H;
  q.npair = (q.dh + 1) / 2;
  st = choose_path(&q);
  if (st != CAT_OK) return st;
  if (q.path == cat::PATH_FAST) {
    q.use_graph = 1;
    if (const char* g = std::getenv("CAT_GRAPH")) q.use_graph = std::strcmp(g, "0") != 0;
  }
  q.workspace_bytes = planned_workspace(&q);
  if (workspace_bytes) *workspace_bytes = q.workspace_bytes;
  if (desc && len > 0) {
    describe(&q);
    std::snprintf(desc, (size_t)len, "%s", q.desc);
  }
  return CAT_OK;
}

int cat_plan_destroy(cat_plan_t plan) {
  if (!plan) return CAT_OK;
  int dev = -1;
  const int plan_dev = plan->device;
  cudaGetDevice(&dev);
  if (dev != plan_dev) cudaSetDevice(plan_dev);
  cudaError_t e = cudaStreamSynchronize(plan->stream);
  free_plan(plan);
  if (dev >= 0 && dev != plan_dev) cudaSetDevice(dev);
  return map_cuda(e);
}

int cat_plan_set_stream(cat_plan_t plan, void* stream) {
  if (!plan) return CAT_ERR_INVALID_ARG;
  plan->stream = (cudaStream_t)stream;
  return CAT_OK;
}

int cat_forward(cat_plan_t p, const void* X, const void* WA, const void* V, void* O, int B, int N,
                int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !V || !O) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WA | (uintptr_t)V | (uintptr_t)O) & 15) return CAT_ERR_MISALIGNED;
  const size_t es = dtype == CAT_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * N * D * es, nw = (size_t)D * H * es;
  if (ranges_overlap(O, nx, X, nx) || ranges_overlap(O, nx, WA, nw) || ranges_overlap(O, nx, V, nx))
    return CAT_ERR_ALIAS;
  cudaEvent_t* ev = nullptr;
  if (p->timing_n < p->timing_cap) ev = p->ev + (size_t)p->ev_per_call * p->timing_n++;
  if (!ev && p->use_graph) {
    const cudaError_t e = launch_forward_graph(p, X, WA, V, O);
    if (e == cudaSuccess) return CAT_OK;
    // Capture or instantiation failed: clear the error and launch the same
    // schedule directly from now on.
    cudaGetLastError();
    p->use_graph = 0;
    describe(p);
  }
  if (!ev && p->path == cat::PATH_FAST) return map_cuda(run_fast_overlapped(p, X, WA, V, O));
  if (ev) cudaEventRecord(ev[0], p->stream);
  if (p->path == cat::PATH_DIRECT) {
    // Scores (in the kernel when fused), softmax and the direct product.
    cudaError_t e = p->dir.fused ? cudaSuccess : cat::launch_score(p, X, WA);
    if (ev) cudaEventRecord(ev[1], p->stream);
    if (ev) cudaEventRecord(ev[2], p->stream);
    if (e == cudaSuccess) e = cat::launch_direct(p, X, WA, V, O, p->dir.fused != 0);
    if (ev) cudaEventRecord(ev[3], p->stream);
    return map_cuda(e);
  }
  cudaError_t e = cat::launch_score(p, X, WA);
  if (e != cudaSuccess) return CAT_ERR_CUDA;
  if (ev) cudaEventRecord(ev[1], p->stream);
  e = p->path == cat::PATH_SMEM   ? cat::launch_softmax_spectrum(p)
      : p->path == cat::PATH_FAST ? cat::launch_fast_zspec(p, 0, p->B * p->H, p->stream, !ev)
                                  : cat::launch_softmax(p);
  if (e != cudaSuccess) return CAT_ERR_CUDA;
  if (ev) cudaEventRecord(ev[2], p->stream);
  if (p->path == cat::PATH_FAST) {
    // Events after each pass of each chunk; the last one closes the stage.
    e = cat::launch_fast_conv(p, V, O, ev ? ev + 3 : nullptr);
  } else {
    e = p->path == cat::PATH_SMEM ? cat::launch_conv_smem(p, V, O)
                                  : cat::launch_fourstep_conv(p, V, O);
    if (ev) cudaEventRecord(ev[3], p->stream);
  }
  return map_cuda(e);
}

namespace {

// Argument checks of the fused projection (bf16, D % 64 == 0, H <= 16,
// 16-byte alignment, V not overlapping the inputs) and the first call's
// workspace for the transposed weights.
int project_prepare(cat_plan_s* p, const void* X, const void* WV, const void* WA, const void* V,
                    int B, int N, int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (dtype != CAT_BF16 || D % 64 != 0 || H > 16) return CAT_ERR_INVALID_ARG;
  if (B == 0) return CAT_OK;
  if (!X || !WV || !WA || !V) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WV | (uintptr_t)WA | (uintptr_t)V) & 15) return CAT_ERR_MISALIGNED;
  const size_t nx = (size_t)B * N * D * 2;
  if (ranges_overlap(V, nx, X, nx) || ranges_overlap(V, nx, WV, (size_t)D * D * 2) ||
      ranges_overlap(V, nx, WA, (size_t)D * H * 2))
    return CAT_ERR_ALIAS;
  if (!p->pj_wt) {
    if (cudaMalloc(&p->pj_wt, cat::project_workspace_bytes(D)) != cudaSuccess) {
      cudaGetLastError();
      p->pj_wt = nullptr;
      return CAT_ERR_ALLOC;
    }
    if (cat::setup_project_kernels() != cudaSuccess) {
      cudaGetLastError();
      return CAT_ERR_CUDA;
    }
  }
  return CAT_OK;
}

}  // namespace

// The fused-projection forward: V = X·W_V and the scores in one pass over X
// on the tensor cores, then the plan's own softmax, spectrum and circulant
// product on that V (the fast path's overlapped schedule runs without a
// graph here).
int cat_forward_fused(cat_plan_t p, const void* X, const void* WV, const void* WA, void* V,
                      void* O, int B, int N, int D, int H, int dtype) {
  int st = project_prepare(p, X, WV, WA, V, B, N, D, H, dtype);
  if (st != CAT_OK || B == 0) return st;
  if (!O) return CAT_ERR_INVALID_ARG;
  if ((uintptr_t)O & 15) return CAT_ERR_MISALIGNED;
  const size_t nx = (size_t)B * N * D * 2;
  if (ranges_overlap(O, nx, X, nx) || ranges_overlap(O, nx, WV, (size_t)D * D * 2) ||
      ranges_overlap(O, nx, WA, (size_t)D * H * 2) || ranges_overlap(O, nx, V, nx))
    return CAT_ERR_ALIAS;
  cudaError_t e = cat::launch_project(p, X, WV, WA, V, p->pj_wt);
  if (e != cudaSuccess) return CAT_ERR_CUDA;
  switch (p->path) {
    case cat::PATH_FAST:
      e = run_fast_overlapped(p, X, WA, V, O, false);
      break;
    case cat::PATH_SMEM:
      e = cat::launch_softmax_spectrum(p);
      if (e == cudaSuccess) e = cat::launch_conv_smem(p, V, O);
      break;
    case cat::PATH_DIRECT:
      e = cat::launch_direct(p, X, WA, V, O, false);
      break;
    default:
      e = cat::launch_softmax(p);
      if (e == cudaSuccess) e = cat::launch_fourstep_conv(p, V, O);
      break;
  }
  return map_cuda(e);
}

// The fused projection alone: V and, after the softmax, z* (fp32 [B, H, N]).
int cat_project(cat_plan_t p, const void* X, const void* WV, const void* WA, void* V,
                float* zstar, int B, int N, int D, int H, int dtype) {
  int st = project_prepare(p, X, WV, WA, V, B, N, D, H, dtype);
  if (st != CAT_OK || B == 0) return st;
  if (!zstar) return CAT_ERR_INVALID_ARG;
  if ((uintptr_t)zstar & 15) return CAT_ERR_MISALIGNED;
  const size_t nx = (size_t)B * N * D * 2, nz = (size_t)B * H * N * sizeof(float);
  if (ranges_overlap(zstar, nz, X, nx) || ranges_overlap(zstar, nz, V, nx))
    return CAT_ERR_ALIAS;
  cudaError_t e = cat::launch_project(p, X, WV, WA, V, p->pj_wt);
  if (e == cudaSuccess)
    e = p->path == cat::PATH_SMEM ? cat::launch_softmax_spectrum(p) : cat::launch_softmax(p);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(zstar, p->zs, nz, cudaMemcpyDeviceToDevice, p->stream);
  return map_cuda(e);
}

int cat_forward_zstar(cat_plan_t p, const void* X, const void* WA, float* zstar, int B, int N,
                      int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !zstar) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WA | (uintptr_t)zstar) & 15) return CAT_ERR_MISALIGNED;
  st = run_front(p, X, WA);
  if (st != CAT_OK) return st;
  return map_cuda(cudaMemcpyAsync(zstar, p->zs, (size_t)B * H * N * sizeof(float),
                                  cudaMemcpyDeviceToDevice, p->stream));
}

namespace {

// Set-up of the host-buffer path at its first call (see cat_plan_s).
int ensure_host(cat_plan_s* p) {
  if (p->hready) return CAT_OK;
  const size_t es = p->dtype == CAT_BF16 ? 2 : 4;
  // CAT_HOST_PIPELINE=0: the serial copy, compute, copy (for comparison).
  const char* pipe = std::getenv("CAT_HOST_PIPELINE");
  const bool steps = p->B >= 2 && !(pipe && std::strcmp(pipe, "0") == 0);
  const size_t nx = (size_t)(steps ? 1 : p->B) * p->N * p->D * es;
  const size_t nw = (size_t)p->D * p->H * es;
  bool ok = cudaMalloc(&p->hwa, nw) == cudaSuccess;
  for (int k = 0; k < (steps ? 2 : 1) && ok; ++k)
    ok = cudaMalloc(&p->hx[k], nx) == cudaSuccess && cudaMalloc(&p->hv[k], nx) == cudaSuccess &&
         cudaMalloc(&p->ho[k], nx) == cudaSuccess;
  int st = ok ? CAT_OK : CAT_ERR_ALLOC;
  if (st == CAT_OK && steps) {
    for (int k = 0; k < 2 && st == CAT_OK; ++k) {
      st = create_plan(&p->hsub[k], 1, p->N, p->D, p->H, p->dtype, p->stream, 0, 0);
      if (st == CAT_OK &&
          (cudaStreamCreateWithFlags(&p->hcp[k], cudaStreamNonBlocking) != cudaSuccess ||
           cudaEventCreateWithFlags(&p->hev_in[k], cudaEventDisableTiming) != cudaSuccess ||
           cudaEventCreateWithFlags(&p->hev_done[k], cudaEventDisableTiming) != cudaSuccess ||
           cudaEventCreateWithFlags(&p->hev_out[k], cudaEventDisableTiming) != cudaSuccess))
        st = CAT_ERR_CUDA;
    }
  }
  if (st != CAT_OK) {
    cudaGetLastError();
    for (int k = 0; k < 2; ++k) {
      cudaFree(p->hx[k]); cudaFree(p->hv[k]); cudaFree(p->ho[k]);
      p->hx[k] = p->hv[k] = p->ho[k] = nullptr;
      if (p->hsub[k]) free_plan(p->hsub[k]);
      p->hsub[k] = nullptr;
      if (p->hcp[k]) cudaStreamDestroy(p->hcp[k]);
      if (p->hev_in[k]) cudaEventDestroy(p->hev_in[k]);
      if (p->hev_done[k]) cudaEventDestroy(p->hev_done[k]);
      if (p->hev_out[k]) cudaEventDestroy(p->hev_out[k]);
      p->hcp[k] = nullptr;
      p->hev_in[k] = p->hev_done[k] = p->hev_out[k] = nullptr;
    }
    cudaFree(p->hwa);
    p->hwa = nullptr;
    return st;
  }
  p->hready = 1;
  return CAT_OK;
}

}  // namespace

// With two or more batches the call runs one batch per step: the inputs of
// step b go in on the first copy stream while step b - 1 computes on the
// plan's stream and step b - 2's output comes back on the second, so the
// host-to-device and device-to-host copies overlap each other and the
// compute.  Step b uses staging slot b mod 2 and that slot's one-batch
// sub-plan; events make a slot's input copy wait for the compute two steps
// back, and its compute wait for its inputs and for the output copy two
// steps back.
int cat_forward_host(cat_plan_t p, const void* X, const void* WA, const void* V, void* O, int B,
                     int N, int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !V || !O) return CAT_ERR_INVALID_ARG;
  const size_t es = dtype == CAT_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * N * D * es, nw = (size_t)D * H * es;
  st = ensure_host(p);
  if (st != CAT_OK) return st;
  if (!p->hsub[0]) {
    cudaError_t e = cudaMemcpyAsync(p->hx[0], X, nx, cudaMemcpyHostToDevice, p->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->hwa, WA, nw, cudaMemcpyHostToDevice, p->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->hv[0], V, nx, cudaMemcpyHostToDevice, p->stream);
    if (e != cudaSuccess) return CAT_ERR_CUDA;
    st = cat_forward(p, p->hx[0], p->hwa, p->hv[0], p->ho[0], B, N, D, H, dtype);
    if (st != CAT_OK) return st;
    e = cudaMemcpyAsync(O, p->ho[0], nx, cudaMemcpyDeviceToHost, p->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
    return map_cuda(e);
  }
  const size_t nb = (size_t)N * D * es;
  const char* xs = static_cast<const char*>(X);
  const char* vs = static_cast<const char*>(V);
  char* os = static_cast<char*>(O);
  cudaStream_t in = p->hcp[0], out = p->hcp[1];
  // W_A first on the input stream: every step's compute waits for an event
  // recorded after it there.
  cudaError_t e = cudaStreamWaitEvent(in, p->hev_done[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(in, p->hev_done[1], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->hwa, WA, nw, cudaMemcpyHostToDevice, in);
  for (int b = 0; b < B && e == cudaSuccess; ++b) {
    const int s = b & 1;
    cat_plan_s* sub = p->hsub[s];
    sub->stream = p->stream;
    e = cudaStreamWaitEvent(in, p->hev_done[s], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->hx[s], xs + b * nb, nb, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->hv[s], vs + b * nb, nb, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess) e = cudaEventRecord(p->hev_in[s], in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->stream, p->hev_in[s], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->stream, p->hev_out[s], 0);
    if (e != cudaSuccess) break;
    st = cat_forward(sub, p->hx[s], p->hwa, p->hv[s], p->ho[s], 1, N, D, H, dtype);
    if (st != CAT_OK) return st;
    e = cudaEventRecord(p->hev_done[s], p->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(out, p->hev_done[s], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(os + b * nb, p->ho[s], nb, cudaMemcpyDeviceToHost, out);
    if (e == cudaSuccess) e = cudaEventRecord(p->hev_out[s], out);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(out);
  return map_cuda(e);
}

namespace {

// The backward's schedule: score, softmax, the correlation and the softmax
// backward (dz* and dz), then dW_A, dX and dV = circ(z*)^T dO, the forward's
// own spectrum and product on the scores reversed.  On the fast path with
// N2 = 32 the reversed scores' spectrum comes first and every correlation
// chunk finishes its rows of dV from its own transform of dO; on the other
// fast shapes dV runs the forward's overlapped schedule with dW_A and dX
// (which need only dz) on the plan's stream beside its chunks.
cudaError_t backward_schedule(cat_plan_s* p, const void* X, const void* WA, const void* V,
                              const void* dO, void* dX, void* dWA, void* dV) {
  if (p->path == cat::PATH_FAST && cat::backward_dv_in_corr(p)) {
    // z* (zs) and its spectrum from the row spectrum kernel, so that the
    // correlation's chunks give dV from their own transform of dO (pass B
    // with the spectrum conjugated: that of z* reversed); dW_A and dX once
    // dz is complete.
    cudaError_t e = cat::launch_score(p, X, WA);
    if (e == cudaSuccess) e = cat::launch_fast_zspec(p, 0, p->B * p->H, p->stream, true, p->zs);
    if (e == cudaSuccess) e = cat::launch_backward_dz(p, dO, V, dV);
    if (e == cudaSuccess) e = cat::launch_backward_dense(p, X, WA, dX, dWA);
    const cudaError_t ej = cat::backward_join_dv(p);   // also after an error: close the fork
    return e == cudaSuccess ? ej : e;
  }
  if (p->path == cat::PATH_SMEM && p->sm.reg_m && !p->twod) {
    // Register path: one spectrum kernel gives z* (for the softmax
    // backward) and FFT(z*)/N.  circ(z*)^T = circ(r) with r[n] = z*[(-n)
    // mod N], and z* is real, so FFT(r) = conj(FFT(z*)): the product kernel
    // takes the spectrum conjugated, with no second softmax and spectrum of
    // the scores reversed.
    cudaError_t e = cat::launch_score(p, X, WA);
    if (e == cudaSuccess) e = cat::launch_softmax_spectrum(p);
    if (e == cudaSuccess) e = cat::launch_backward_dz(p, dO, V);
    if (e == cudaSuccess) e = cat::launch_backward_dense(p, X, WA, dX, dWA);
    if (e == cudaSuccess) e = cat::launch_conv_reg(p, dO, dV, true);
    return e;
  }
  if (run_backward_front(p, X, WA, V, dO) != CAT_OK) return cudaErrorLaunchFailure;
  if (p->path == cat::PATH_FAST) {
    cudaError_t e = cat::launch_reverse_scores(p);
    const std::function<cudaError_t()> dense = [&]() {
      return cat::launch_backward_dense(p, X, WA, dX, dWA);
    };
    if (e == cudaSuccess) e = run_fast_overlapped(p, nullptr, nullptr, dO, dV, false, &dense);
    return e;
  }
  cudaError_t e = cat::launch_backward_dense(p, X, WA, dX, dWA);
  if (e == cudaSuccess) e = cat::launch_reverse_scores(p);
  if (e != cudaSuccess) return e;
  if (p->path == cat::PATH_SMEM) {
    e = cat::launch_softmax_spectrum(p);
    if (e == cudaSuccess) e = cat::launch_conv_smem(p, dO, dV);
  } else if (p->path == cat::PATH_DIRECT) {
    e = cat::launch_direct(p, nullptr, nullptr, dO, dV, false);
  } else {
    e = cat::launch_softmax(p);
    if (e == cudaSuccess) e = cat::launch_fourstep_conv(p, dO, dV);
  }
  return e;
}

// The same schedule through a CUDA graph, captured on the private stream
// as the forward's is, and replayed while the call's pointers stay the same.
cudaError_t launch_backward_graph(cat_plan_s* p, const void* X, const void* WA, const void* V,
                                  const void* dO, void* dX, void* dWA, void* dV) {
  const void* ptrs[7] = {X, WA, V, dO, dX, dWA, dV};
  bool same = p->bgexec != nullptr;
  for (int k = 0; k < 7 && same; ++k) same = ptrs[k] == p->bgp[k];
  if (!same) {
    cudaStream_t saved = p->stream;
    p->stream = p->cap;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      const cudaError_t e1 = backward_schedule(p, X, WA, V, dO, dX, dWA, dV);
      const cudaError_t e2 = cudaStreamEndCapture(p->cap, &g);
      e = e1 != cudaSuccess ? e1 : e2;
    }
    p->stream = saved;
    if (e == cudaSuccess && p->bgexec) {
      cudaGraphExecUpdateResultInfo info;
      if (cudaGraphExecUpdate(p->bgexec, g, &info) != cudaSuccess) {
        cudaGetLastError();
        cudaGraphExecDestroy(p->bgexec);
        p->bgexec = nullptr;
      }
    }
    if (e == cudaSuccess && !p->bgexec) e = cudaGraphInstantiate(&p->bgexec, g, 0);
    if (g) cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      if (p->bgexec) cudaGraphExecDestroy(p->bgexec);
      p->bgexec = nullptr;
      return e;
    }
    for (int k = 0; k < 7; ++k) p->bgp[k] = ptrs[k];
  }
  return cudaGraphLaunch(p->bgexec, p->stream);
}

}  // namespace

int cat_backward(cat_plan_t p, const void* X, const void* WA, const void* V, const void* dO,
                 void* dX, void* dWA, void* dV, int B, int N, int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !V || !dO || !dX || !dWA || !dV) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WA | (uintptr_t)V | (uintptr_t)dO | (uintptr_t)dX |
       (uintptr_t)dWA | (uintptr_t)dV) & 15)
    return CAT_ERR_MISALIGNED;
  const size_t es = dtype == CAT_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * N * D * es, nw = (size_t)D * H * es;
  const void* in[4] = {X, WA, V, dO};
  const size_t in_n[4] = {nx, nw, nx, nx};
  const void* out[3] = {dX, dWA, dV};
  const size_t out_n[3] = {nx, nw, nx};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 4; ++i)
      if (ranges_overlap(out[o], out_n[o], in[i], in_n[i])) return CAT_ERR_ALIAS;
    for (int q = o + 1; q < 3; ++q)
      if (ranges_overlap(out[o], out_n[o], out[q], out_n[q])) return CAT_ERR_ALIAS;
  }
  st = ensure_backward(p);
  if (st != CAT_OK) return st;
  if (p->use_graph) {
    const cudaError_t e = launch_backward_graph(p, X, WA, V, dO, dX, dWA, dV);
    if (e == cudaSuccess) return CAT_OK;
    // Capture or instantiation failed: clear the error and launch the
    // schedule directly from now on.
    cudaGetLastError();
    p->use_graph = 0;
    describe(p);
  }
  return map_cuda(backward_schedule(p, X, WA, V, dO, dX, dWA, dV));
}

int cat_backward_dz(cat_plan_t p, const void* X, const void* WA, const void* V, const void* dO,
                    float* dzstar, float* dz, int B, int N, int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (p->twod) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !V || !dO || !dzstar || !dz) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WA | (uintptr_t)V | (uintptr_t)dO | (uintptr_t)dzstar |
       (uintptr_t)dz) & 15)
    return CAT_ERR_MISALIGNED;
  {
    const size_t es = dtype == CAT_BF16 ? 2 : 4;
    const size_t nx = (size_t)B * N * D * es, nw = (size_t)D * H * es;
    const size_t nz = (size_t)B * H * N * sizeof(float);
    const void* in[4] = {X, WA, V, dO};
    const size_t in_n[4] = {nx, nw, nx, nx};
    for (int i = 0; i < 4; ++i)
      if (ranges_overlap(dzstar, nz, in[i], in_n[i]) || ranges_overlap(dz, nz, in[i], in_n[i]))
        return CAT_ERR_ALIAS;
    if (ranges_overlap(dzstar, nz, dz, nz)) return CAT_ERR_ALIAS;
  }
  st = ensure_backward(p);
  if (st != CAT_OK) return st;
  st = run_backward_front(p, X, WA, V, dO);
  if (st != CAT_OK) return st;
  const size_t bytes = (size_t)B * H * N * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(dzstar, p->bw_dzs, bytes, cudaMemcpyDeviceToDevice, p->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dz, p->bw_dz, bytes, cudaMemcpyDeviceToDevice, p->stream);
  return map_cuda(e);
}

int cat2d_scores(cat_plan_t p, const void* Q, const void* K, float* a, int B, int h, int w, int D,
                 int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (!p->twod || h != p->grid_h || w != p->grid_w) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, h * w, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!Q || !K || !a) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)Q | (uintptr_t)K | (uintptr_t)a) & 15) return CAT_ERR_MISALIGNED;
  const size_t nx = (size_t)B * p->N * D * (dtype == CAT_BF16 ? 2 : 4);
  const size_t na = (size_t)B * H * p->N * sizeof(float);
  if (ranges_overlap(a, na, Q, nx) || ranges_overlap(a, na, K, nx)) return CAT_ERR_ALIAS;
  if (p->gp2d) return map_cuda(cat::launch_grid_pass(p, Q, K, nullptr, nullptr, a));
  return map_cuda(p->reg2d ? cat::launch_scores2d_reg(p, Q, K, a) : cat::launch_scores2d(p, Q, K, a));
}

int cat2d_forward(cat_plan_t p, const void* Q, const void* K, const void* V, void* O, int B,
                  int h, int w, int D, int H, int dtype) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (!p->twod || h != p->grid_h || w != p->grid_w) return CAT_ERR_PLAN_MISMATCH;
  int st = check_shape(p, B, h * w, D, H, dtype);
  if (st != CAT_OK) return st;
  if (B == 0) return CAT_OK;
  if (!Q || !K || !V || !O) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)Q | (uintptr_t)K | (uintptr_t)V | (uintptr_t)O) & 15) return CAT_ERR_MISALIGNED;
  const size_t es = dtype == CAT_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * p->N * D * es;
  if (ranges_overlap(O, nx, Q, nx) || ranges_overlap(O, nx, K, nx) || ranges_overlap(O, nx, V, nx))
    return CAT_ERR_ALIAS;
  if (p->gp2d) return map_cuda(cat::launch_grid_pass(p, Q, K, V, O, nullptr));
  if (p->reg2d) {
    // Register kernels: scores, softmax with the 2-D spectrum, product.
    cudaError_t e = cat::launch_scores2d_reg(p, Q, K, nullptr);
    if (e == cudaSuccess) e = cat::launch_softmax_spectrum_reg(p);
    if (e == cudaSuccess) e = cat::launch_conv_reg(p, V, O);
    return map_cuda(e);
  }
  cudaError_t e = cat::launch_scores2d(p, Q, K);
  if (e == cudaSuccess) e = cat::launch_softmax(p);
  if (e == cudaSuccess) e = cat::launch_fourstep_conv(p, V, O);
  return map_cuda(e);
}

int cat_plan_sync(cat_plan_t p) {
  if (!p) return CAT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(p->stream) != cudaSuccess) return CAT_ERR_CUDA;
  // The plan's own status word and those of its host-buffer sub-plans.
  int st = CAT_OK;
  for (cat_plan_s* q : {p, p->hsub[0], p->hsub[1]}) {
    if (!q) continue;
    unsigned int word = 0;
    if (cudaMemcpy(&word, q->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
      return CAT_ERR_CUDA;
    if (word != 0) {
      if (std::getenv("CAT_LOG")) std::fprintf(stderr, "[cat] device status 0x%x\n", word);
      cudaMemset(q->status, 0, sizeof(unsigned int));
      st = CAT_ERR_DEVICE_STATUS;
    }
  }
  return st;
}

int cat_plan_timing(cat_plan_t p, int max_calls) {
  if (!p || max_calls < 0) return CAT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(p->stream) != cudaSuccess) return CAT_ERR_CUDA;
  free_events(p);
  if (max_calls == 0) return CAT_OK;
  p->ev_per_call = p->path == cat::PATH_FAST ? 3 + 3 * cat::fast_chunks(p) : 4;
  const size_t n = (size_t)p->ev_per_call * max_calls;
  p->ev = new (std::nothrow) cudaEvent_t[n]();
  if (!p->ev) return CAT_ERR_ALLOC;
  p->timing_cap = max_calls;
  for (size_t i = 0; i < n; ++i) {
    if (cudaEventCreate(&p->ev[i]) != cudaSuccess) {
      free_events(p);
      return CAT_ERR_CUDA;
    }
  }
  return CAT_OK;
}

int cat_plan_stage_times(cat_plan_t p, float* ms, int cap, int* ncalls) {
  if (!p || !ms || cap < 3) return CAT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(p->stream) != cudaSuccess) return CAT_ERR_CUDA;
  ms[0] = ms[1] = ms[2] = 0.f;
  for (int c = 0; c < p->timing_n; ++c) {
    cudaEvent_t* ev = p->ev + (size_t)p->ev_per_call * c;
    const int b[4] = {0, 1, 2, p->ev_per_call - 1};
    for (int s = 0; s < 3; ++s) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[b[s]], ev[b[s + 1]]) != cudaSuccess) return CAT_ERR_CUDA;
      ms[s] += t;
    }
  }
  if (ncalls) *ncalls = p->timing_n;
  return CAT_OK;
}

int cat_plan_pass_times(cat_plan_t p, float* ms, int cap, int* launches) {
  if (!p || !ms || cap < 3) return CAT_ERR_INVALID_ARG;
  if (p->path != cat::PATH_FAST) return CAT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(p->stream) != cudaSuccess) return CAT_ERR_CUDA;
  ms[0] = ms[1] = ms[2] = 0.f;
  const int chunks = (p->ev_per_call - 3) / 3;
  for (int c = 0; c < p->timing_n; ++c) {
    cudaEvent_t* ev = p->ev + (size_t)p->ev_per_call * c;
    for (int k = 0; k < chunks; ++k)
      for (int s = 0; s < 3; ++s) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, ev[2 + 3 * k + s], ev[3 + 3 * k + s]) != cudaSuccess)
          return CAT_ERR_CUDA;
        ms[s] += t;
      }
  }
  if (launches) *launches = p->timing_n * chunks;
  return CAT_OK;
}

int cat_plan_describe(cat_plan_t p, char* buf, int len) {
  if (!p || !buf || len <= 0) return CAT_ERR_INVALID_ARG;
  std::snprintf(buf, (size_t)len, "%s", p->desc);
  return CAT_OK;
}

const char* cat_status_string(int status) {
  switch (status) {
    case CAT_OK: return "CAT_OK";
    case CAT_ERR_INVALID_ARG: return "CAT_ERR_INVALID_ARG";
    case CAT_ERR_UNSUPPORTED_N: return "CAT_ERR_UNSUPPORTED_N";
    case CAT_ERR_MISALIGNED: return "CAT_ERR_MISALIGNED";
    case CAT_ERR_PLAN_MISMATCH: return "CAT_ERR_PLAN_MISMATCH";
    case CAT_ERR_ALLOC: return "CAT_ERR_ALLOC";
    case CAT_ERR_CUDA: return "CAT_ERR_CUDA";
    case CAT_ERR_DEVICE_STATUS: return "CAT_ERR_DEVICE_STATUS";
    case CAT_ERR_ALIAS: return "CAT_ERR_ALIAS";
    case CAT_ERR_TOO_LARGE: return "CAT_ERR_TOO_LARGE";
    default: return "CAT_ERR_UNKNOWN";
  }
}

}  // extern "C"
