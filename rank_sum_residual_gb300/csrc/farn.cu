// Host side of libfarn.so: the C ABI declared in include/farn.h.
//
// Argument checks, the choice of kernel variant for a shape, and the launch
// on the caller's stream.  The page's host side (FlagTree pull request
// "[TLERaw] Add NVSHMEM allreduce RMSNorm tutorial", Implementation
// section 4) initialises NVSHMEM, bootstraps the ranks and manages a
// symmetric workspace behind a host C ABI; on one GPU none of that exists,
// so the context only caches device properties and kernel attributes, and
// the library allocates no device memory at all.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "farn.h"
#include "farn_kernels.cuh"

static_assert(FARN_MAX_W == farn::kMaxW, "FARN_MAX_W and kernel limit differ");

enum {
  kVariantRow = 0,
  kVariantCluster = 1,
  kVariantGeneric = 2,
  kVariantBulk = 3,
  kVariantStage = 4,
  kVariantCombine = 5,   // the MoE combine's one-CTA-per-row gather kernel
  kVariantAuto = -1
};

struct farn_ctx {
  int device;
  int num_sms;
  int max_cluster;     // largest power-of-two cluster size that can be scheduled
  int force_variant;   // kVariantAuto unless FARN_VARIANT says otherwise
  int force_cluster;   // 0 = choose; else CTAs per row for the cluster variant
  int force_vpt;       // 0 = choose; else 16-byte vectors per thread
  int pdl;             // launch with programmatic stream serialisation
  int64_t small_t;     // below this many rows a call counts as latency bound
  int bulk;            // 1: the TMA-staged kernel serves long inputs by default
  int bulk_ctas;       // resident bulk CTAs per SM (1 or 2)
  int stage;           // 1: the cp.async-staged kernel serves long inputs
  int stage_r;         // 0 = choose; else chunks in flight per thread (8/12/16)
  int stage_ctas;      // 0 = choose; else resident stage CTAs per SM (1..4)
  int64_t stage_min_t; // the stage kernel serves calls with at least this many rows,
  int64_t stage_min_bytes;  // or half as many that read at least this many bytes
  int stage_regs[4][2];  // registers per thread of the staged kernels
                         // [plain, FP8, MoE combine, NVFP4][4 vectors]
  int max_smem;        // opt-in shared memory per CTA, bytes
  int* d_status;       // device status word of the bulk kernel (256 B block)
  int fault_launch;    // FARN_FAULT_INJECT=launch at create: every launch fails
  int stall_test;      // FARN_FAULT_INJECT=stall at create: the TMA-staged kernel's
                       // CTA 0 runs its bounded waits out (a test of the status word)
};

namespace {

typedef void (*VecKernel)(const farn::Params);

// Chunks in flight per thread that the stage kernels are built for (the
// FP8- and NVFP4-output kernels also at 6, so that two of their CTAs share
// an SM at H = 8192).
constexpr int kStageDepths[4] = {16, 12, 8, 6};

// Quantised copy of norm_out written alongside (the stage kernel's QM).
enum { kQuantNone = 0, kQuantFp8 = 1, kQuantNvfp4 = 2 };

template <int QM>
VecKernel pick_stage_q(int vpt, int r) {
  if (vpt == 2) {
    if (r == 8) return &farn::farn_stage_kernel<2, 8, QM>;
    if (r == 12) return &farn::farn_stage_kernel<2, 12, QM>;
    if (r == 16) return &farn::farn_stage_kernel<2, 16, QM>;
    if constexpr (QM != kQuantNone)
      if (r == 6) return &farn::farn_stage_kernel<2, 6, QM>;
  } else if (vpt == 4) {
    if (r == 8) return &farn::farn_stage_kernel<4, 8, QM>;
    if (r == 12) return &farn::farn_stage_kernel<4, 12, QM>;
    if (r == 16) return &farn::farn_stage_kernel<4, 16, QM>;
    if constexpr (QM != kQuantNone)
      if (r == 6) return &farn::farn_stage_kernel<4, 6, QM>;
  }
  return nullptr;
}

// qm: the instantiation that also writes the FP8 or the NVFP4 output
VecKernel pick_stage(int vpt, int r, int qm = kQuantNone) {
  return qm == kQuantFp8     ? pick_stage_q<kQuantFp8>(vpt, r)
         : qm == kQuantNvfp4 ? pick_stage_q<kQuantNvfp4>(vpt, r)
                             : pick_stage_q<kQuantNone>(vpt, r);
}

VecKernel pick_combine_stage(int vpt, int r) {
  if (vpt == 2) {
    if (r == 8) return &farn::farn_combine_stage_kernel<2, 8>;
    if (r == 12) return &farn::farn_combine_stage_kernel<2, 12>;
    if (r == 16) return &farn::farn_combine_stage_kernel<2, 16>;
  } else if (vpt == 4) {
    if (r == 8) return &farn::farn_combine_stage_kernel<4, 8>;
    if (r == 12) return &farn::farn_combine_stage_kernel<4, 12>;
    if (r == 16) return &farn::farn_combine_stage_kernel<4, 16>;
  }
  return nullptr;
}

VecKernel pick_generic(int pb) {
  return pb == 4 ? &farn::farn_generic_kernel<4> : &farn::farn_generic_kernel<2>;
}

// The bulk kernel instantiations: the most segments per row each takes.
constexpr int kBulkVpts[5] = {1, 2, 4, 8, 16};

template <bool COMBINE>
VecKernel pick_bulk_t(int vpt) {
  switch (vpt) {
    case 1: return &farn::farn_bulk_kernel<1, COMBINE>;
    case 2: return &farn::farn_bulk_kernel<2, COMBINE>;
    case 4: return &farn::farn_bulk_kernel<4, COMBINE>;
    case 8: return &farn::farn_bulk_kernel<8, COMBINE>;
    case 16: return &farn::farn_bulk_kernel<16, COMBINE>;
  }
  return nullptr;
}

// combine: the MoE combine's instantiation
VecKernel pick_bulk(int vpt, bool combine = false) {
  return combine ? pick_bulk_t<true>(vpt) : pick_bulk_t<false>(vpt);
}

struct Plan {
  int variant;
  int pb;       // bytes per partial element
  int cs;       // CTAs per row
  int vpt;      // vectors per thread
  int threads;  // threads per CTA
  bool one_row; // row/cluster kernel: the one-row (latency-bound) instantiation
  int64_t grid;
  int stage_r;            // stage: chunks in flight per thread
  uint32_t stages;        // bulk: ring stages
  uint32_t stage_stride;  // bulk: bytes per stage
  size_t smem;            // bulk: dynamic shared memory bytes
};

// Bulk plan.  A row of hv vectors is cut into nseg segments of nct
// vectors (nct consumer threads, a multiple of 32, at most 256); a ring
// stage holds one segment of all W+1 inputs.  Chosen: the fewest segments
// per row (fewest waits) whose ring holds at least 4 stages, else the
// deepest ring of at least 2 stages; `ctas` resident CTAs per SM share the
// SM's shared memory.  Where the consumers set the pace -- the MoE combine
// (combine) and rank sums of W >= 8 inputs -- rows of one or two segments
// may take up to 512 consumer threads, and the fewest segments whose ring
// holds 2 stages win.  Measured on GB300 (T = 8192, H = 4096..8192): at
// W = 8, 95.2-100.3 % of the copy bandwidth with one or two segments of up
// to 512 consumers against 92.3-94.9 % with at most 256 and 4 stages; at
// W = 16, 98.8-104.6 % against 97.2-102.3 %; at W = 4 the other way
// (81.4-89.0 % against 86.2-96.0 %).  Rows longer than kBulkMaxH elements
// are not taken (every shorter row is, for any W <= 32, at one CTA per SM:
// the longest row at W = 32 takes 16 segments of 128 vectors and 3 stages).
// force_vpt (FARN_VPT), when set, caps the segments per row.
bool bulk_fit(const farn_ctx* ctx, int W, int64_t T, int64_t H, int ctas, Plan* pl,
              bool combine) {
  if (H > farn::kBulkMaxH) return false;
  const int64_t hv = H / 8;
  const int max_seg = ctx->force_vpt > 0 ? ctx->force_vpt : 16;
  const size_t budget = (size_t)ctx->max_smem / (size_t)ctas;
  const size_t fixed = sizeof(farn::BulkBarriers) + 128;
  if (budget <= fixed) return false;
  const bool wide = combine || W >= 8;
  int best_seg = 0, best_nct = 0;
  size_t best_ns = 0;
  uint32_t best_stride = 0;
  for (int nseg = 1; nseg <= max_seg; ++nseg) {
    const int64_t nct = ((hv + nseg - 1) / nseg + 31) / 32 * 32;
    if (nct > ((wide && nseg <= 2) ? farn::kBulkMaxConsumersWide : farn::kBulkMaxConsumers))
      continue;
    if ((hv + nct - 1) / nct != nseg) continue;   // the same split as fewer segments
    const uint32_t stride = (uint32_t)((nct * 16 + 127) / 128 * 128);
    size_t ns = (budget - fixed) / ((size_t)(W + 1) * stride);
    if (ns > farn::kBulkMaxStages) ns = farn::kBulkMaxStages;
    if (ns >= (wide ? 2u : 4u)) {
      best_seg = nseg; best_nct = (int)nct; best_ns = ns; best_stride = stride;
      break;
    }
    if (ns >= 2 && ns > best_ns) { best_seg = nseg; best_nct = (int)nct; best_ns = ns; best_stride = stride; }
  }
  if (!best_seg) return false;
  int vpt = 0;
  for (int v : kBulkVpts)
    if (!vpt && v >= best_seg) vpt = v;
  if (!vpt || !pick_bulk(vpt)) return false;
  pl->variant = kVariantBulk;
  pl->pb = 2;
  pl->cs = 1;
  pl->one_row = false;
  pl->vpt = vpt;
  pl->threads = best_nct + 32;
  const int64_t resident = (int64_t)ctx->num_sms * ctas;
  pl->grid = T < resident ? T : resident;
  pl->stages = (uint32_t)best_ns;
  pl->stage_stride = best_stride;
  pl->smem = best_ns * (size_t)(W + 1) * best_stride + sizeof(farn::BulkBarriers);
  return true;
}

// One resident CTA per SM unless FARN_BULK_CTAS=2 (then two where the
// plan fits half the shared memory).  With the producer warp issuing a
// segment's copies from W+1 lanes, one CTA per SM measured fastest on
// GB300 (W = 4, T = 32768, H = 5120: 96.9 % of the copy bandwidth against
// 89.5 % for two; W = 8, T = 8192, H = 8192: 97.0 % against 96.4 %; W = 16,
// T = 4096, H = 7168: 98.7 % against 83.4 %).
bool make_bulk_plan(const farn_ctx* ctx, int W, int64_t T, int64_t H, Plan* pl,
                    bool combine = false) {
  if (ctx->bulk_ctas == 2 && bulk_fit(ctx, W, T, H, 2, pl, combine)) return true;
  return bulk_fit(ctx, W, T, H, 1, pl, combine);
}

template <int VPT, int CS, int PB>
VecKernel vec_kernel() { return &farn::farn_vec_kernel<VPT, CS, PB>; }

template <int PB>
VecKernel pick_vec_pb(int vpt, int cs) {
  switch (cs) {
    case 1:
      switch (vpt) { case 1: return vec_kernel<1, 1, PB>(); case 2: return vec_kernel<2, 1, PB>();
                     case 4: return vec_kernel<4, 1, PB>(); }
      break;
    case 2:
      switch (vpt) { case 1: return vec_kernel<1, 2, PB>(); case 2: return vec_kernel<2, 2, PB>();
                     case 4: return vec_kernel<4, 2, PB>(); }
      break;
    case 4:
      switch (vpt) { case 1: return vec_kernel<1, 4, PB>(); case 2: return vec_kernel<2, 4, PB>();
                     case 4: return vec_kernel<4, 4, PB>(); }
      break;
    case 8:
      switch (vpt) { case 1: return vec_kernel<1, 8, PB>(); case 2: return vec_kernel<2, 8, PB>();
                     case 4: return vec_kernel<4, 8, PB>(); }
      break;
    case 16:
      switch (vpt) { case 1: return vec_kernel<1, 16, PB>(); case 2: return vec_kernel<2, 16, PB>();
                     case 4: return vec_kernel<4, 16, PB>(); }
      break;
  }
  return nullptr;
}

// The one-row instantiations (bf16 partials, one vector per thread) that
// serve latency-bound calls.
template <bool QUANT>
VecKernel pick_vec_one_row_q(int cs) {
  switch (cs) {
    case 1: return &farn::farn_vec_kernel<1, 1, 2, true, QUANT>;
    case 2: return &farn::farn_vec_kernel<1, 2, 2, true, QUANT>;
    case 4: return &farn::farn_vec_kernel<1, 4, 2, true, QUANT>;
    case 8: return &farn::farn_vec_kernel<1, 8, 2, true, QUANT>;
    case 16: return &farn::farn_vec_kernel<1, 16, 2, true, QUANT>;
  }
  return nullptr;
}

// quant: the call writes an FP8 or NVFP4 output (only the one-row builds
// come in two versions; the others always carry that code)
VecKernel pick_vec(int vpt, int cs, int pb, bool one_row = false, bool quant = true) {
  if (one_row) {
    if (vpt != 1 || pb != 2) return nullptr;
    return quant ? pick_vec_one_row_q<true>(cs) : pick_vec_one_row_q<false>(cs);
  }
  return pb == 4 ? pick_vec_pb<4>(vpt, cs) : pick_vec_pb<2>(vpt, cs);
}

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (na <= 0 || nb <= 0) return false;
  uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + (uintptr_t)nb && b0 < a0 + (uintptr_t)na;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int env_int(const char* name, int dflt) {
  const char* s = getenv(name);
  if (!s || !*s) return dflt;
  return atoi(s);
}

// Vectors per thread for a slice of sv 16-byte vectors (the vector kernel
// takes at most 512 threads, so slices of up to 2048 vectors, H <= 16384
// for one CTA per row).
// Below this many rows a latency-bound call splits rows over a cluster.
constexpr int64_t kClusterRowsMax = 16;
// Long calls with at least this many bf16 inputs default to the TMA-staged
// kernel (see make_plan).
constexpr int kBulkDefaultMinW = 12;
constexpr int64_t kBulkDefaultMinT = 256;
// Long calls with fewer bf16 inputs and a bf16 norm_out take the row kernel
// (see make_plan).
constexpr int kStageMinW = 8;
// With kStageMinW <= W < kBulkDefaultMinW the row length decides: rows of at
// most kRowMaxH elements take the row kernel, rows shorter than kStageMinH
// the TMA-staged kernel, longer ones the cp.async-staged kernel.
constexpr int64_t kRowMaxH = 5120;
constexpr int64_t kStageMinH = 8192;

int choose_vpt(int64_t sv) {
  if (sv >= 512) return 4;
  if (sv >= 128) return 2;
  return 1;
}

// Stage plan.  Measured on GB300 (prefill / nonpow2 / wide shapes, and
// H = 2048 / 4096 at T = 1k-8k): what matters is both the bytes each SM
// keeps in flight and having at least two CTAs (or one of 512 threads) per
// SM, so that one row's reduction overlaps another row's loads.  So:
//   1. 4, then 2 vectors per thread (2 first for the FP8 and NVFP4
//      outputs), with the fewest CTAs per SM (2..4) that give >= 320
//      threads per SM and fit registers and shared memory;
//   2. else one CTA per SM, 2 then 4 vectors per thread;
// each with the largest of 16 / 12 / 8 chunks in flight per thread that fits
// (also 6 for the FP8 and NVFP4 outputs).
// kind: 0 plain stage kernel, 1 with the FP8 output, 2 the staged MoE
// combine, 3 with the NVFP4 output
bool stage_fit(const farn_ctx* ctx, int64_t hv, int vpt, int ctas, Plan* pl, int64_t T,
               int kind) {
  const bool quant = kind == 1 || kind == 3;
  const int qm = kind == 1 ? kQuantFp8 : (kind == 3 ? kQuantNvfp4 : kQuantNone);
  if (ctx->force_vpt > 0 && ctx->force_vpt != vpt) return false;
  if (ctx->stage_ctas > 0 && ctx->stage_ctas != ctas) return false;
  const int64_t nt = ((hv + vpt - 1) / vpt + 31) / 32 * 32;
  if (nt > 512) return false;
  const int regs = ctx->stage_regs[kind][vpt >= 4];
  if ((int64_t)regs * nt * ctas > 65536) return false;
  const size_t budget = (size_t)ctx->max_smem / (size_t)ctas - 1024;
  int r = 0;
  for (int i = 0; i < (quant ? 4 : 3) && !r; ++i) {
    const int cand = kStageDepths[i];
    if (ctx->stage_r > 0 && cand != ctx->stage_r) continue;
    if ((size_t)cand * vpt * nt * 16 <= budget) r = cand;
  }
  if (!r || !(kind == 2 ? pick_combine_stage(vpt, r) : pick_stage(vpt, r, qm)))
    return false;
  pl->variant = kVariantStage;
  pl->pb = 2;
  pl->cs = 1;
  pl->one_row = false;
  pl->vpt = vpt;
  pl->threads = (int)nt;
  const int64_t resident = (int64_t)ctx->num_sms * ctas;
  pl->grid = T < resident ? T : resident;
  pl->stage_r = r;
  pl->smem = (size_t)r * vpt * nt * 16;
  return true;
}

// Long enough for the persistent stage kernels: at least stage_min_t rows,
// or half that many when the call reads at least stage_min_bytes.  (GB300,
// T = 1024: the stage kernel 90.8 % / 85.0 % of the copy bandwidth against
// 82.0 % / 80.8 % for the row kernel on the prefill / wide shapes, which
// read 151 / 250 MB; 66.8 % against 71.1 % on nonpow2, 52 MB; at T = 512
// the row kernel is ahead on all three.)
bool long_call(const farn_ctx* ctx, int64_t T, int64_t in_bytes) {
  return T >= ctx->stage_min_t || (T >= ctx->stage_min_t / 2 && in_bytes >= ctx->stage_min_bytes);
}

// bf16 partials only (fp32 partials take the row kernel, see the kernel).
bool make_stage_plan(const farn_ctx* ctx, int64_t T, int64_t H, Plan* pl, int kind) {
  const int64_t hv = H / 8;
  // The quantising kernels and the staged MoE combine try 2 vectors per
  // thread first: at H = 8192 two CTAs of 512 threads (6 chunks in flight)
  // measured 101.0 % (NVFP4) and 95.1 % (FP8) of the copy bandwidth against
  // 96.4 % and 94.8 % for two CTAs of 256 threads at 4 vectors; the combine
  // at H = 7168, K = 8, 89.7 % with two CTAs of 448 threads against 88.3 %
  // with two of 224 at 4 vectors.
  const bool two_first = kind == 1 || kind == 2 || kind == 3;
  const int vpts[2] = {two_first ? 2 : 4, two_first ? 4 : 2};
  if (ctx->stage_ctas > 0)   // a forced CTA count: the first vector count that fits it
    return stage_fit(ctx, hv, vpts[0], ctx->stage_ctas, pl, T, kind) ||
           stage_fit(ctx, hv, vpts[1], ctx->stage_ctas, pl, T, kind);
  for (int i = 0; i < 2; ++i) {
    const int vpt = vpts[i];
    const int64_t nt = ((hv + vpt - 1) / vpt + 31) / 32 * 32;
    int ctas = (int)((320 + nt - 1) / nt);
    if (ctas < 2) ctas = 2;
    for (; ctas <= 4; ++ctas)
      if (stage_fit(ctx, hv, vpt, ctas, pl, T, kind)) return true;
  }
  return stage_fit(ctx, hv, 2, 1, pl, T, kind) || stage_fit(ctx, hv, 4, 1, pl, T, kind);
}

// in_bytes: the bytes the call reads (partials, residual, weight).
int make_plan(const farn_ctx* ctx, int W, int64_t T, int64_t H, bool vec_ok, int pb, Plan* out,
              int qm, int64_t in_bytes) {
  Plan pl;
  pl.pb = pb;
  pl.one_row = false;
  const bool quant = qm != kQuantNone;
  // The FP8 and NVFP4 outputs are produced by every kernel but the
  // TMA-staged one.
  if (quant && ctx->force_variant == kVariantBulk) return FARN_ERR_UNSUPPORTED;
  const int64_t hv = H / 8;
  const int want = ctx->force_variant;
  const bool small = T < ctx->small_t;
  pl.stages = 0; pl.stage_stride = 0; pl.smem = 0;
  // Long calls of W >= 12 bf16 partials (no quantised output) take the
  // TMA-staged kernel.  Measured on GB300 (T = 8192, H = 2048..8192, % of
  // the copy bandwidth, staged against TMA-staged): W = 12..32, 86.3-101.8
  // against 91.8-105.2 %, ahead on 23 of 25 shapes (behind by at most
  // 1.8 points); W = 8, ahead on 3 of 5 (behind by 5.3 points at H = 8192);
  // W = 4 and 6, behind on 6 of 10.
  // With 8..11 partials (T = 8192, % of the copy bandwidth, W = 8 / 10, row /
  // TMA-staged / cp.async-staged): H = 3072..5120 the row kernel leads
  // (95.8-100.6 against 91.9-101.5 / 90.6-92.3); H = 6144 and 7168 the
  // TMA-staged kernel (97.3-105.7 against 90.5-96.7 / 94.2-97.2); H = 8192
  // and above the cp.async-staged kernel (96.7-106.6 against 88.4-100.9 /
  // 96.3-104.8).
  const bool mid_w = W >= kStageMinW && W < kBulkDefaultMinW;
  const bool auto_long = want == kVariantAuto && ctx->force_cluster == 0 && ctx->stage &&
                         long_call(ctx, T, in_bytes);
  // W >= 12 from 256 rows on, below the long-call threshold too (T = 256 /
  // 512, W = 16, % of the copy bandwidth, TMA-staged against row: H = 4096,
  // 61.7 / 77.3 against 51.2 / 77.3; H = 8192, 79.8 / 86.6 against 78.0 /
  // 84.0).
  const bool auto_mid = want == kVariantAuto && ctx->force_cluster == 0 && ctx->stage &&
                        T >= kBulkDefaultMinT;
  const bool bulk_default =
      (auto_mid && W >= kBulkDefaultMinW) ||
      (auto_long && mid_w && H > kRowMaxH && H < kStageMinH);
  const bool bulk_enabled = want == kVariantAuto && ctx->force_cluster == 0 && ctx->bulk && !small;
  if (vec_ok && pb == 2 && !quant &&
      (want == kVariantBulk || bulk_enabled || bulk_default) &&
      make_bulk_plan(ctx, W, T, H, &pl)) {
    *out = pl;
    return FARN_OK;
  }
  if (want == kVariantBulk) return FARN_ERR_UNSUPPORTED;
  pl.stage_r = 0;
  // The cp.async-staged kernel for long calls of 8..11 partials with rows of
  // 8192 elements or more (shorter ones over 5120 took the TMA-staged kernel
  // above) and for the FP8 / NVFP4 outputs; with fewer partials or shorter
  // rows and a bf16 norm_out the row kernel (one CTA per row, the row
  // prefetched into L2 before the dependency wait) streams faster.  Measured on GB300, % of the copy
  // bandwidth, stage against row: nonpow2 (W = 4, T = 32768, H = 5120)
  // 99.4 against 103.1, rmsnorm (W = 1, T = 8192, H = 8192) 95.3 against
  // 98.2; T = 8192, H = 4096..8192: W = 1, 2, 4 behind on all 15 shapes (by
  // 1.6-18.2 points); W = 8 ahead on 2 of 5; prefill (W = 8) 103.8 against
  // 101.0, its FP8 / NVFP4 outputs 101.6 / 100.3 against 96.3 / 92.3.
  // With the FP8 / NVFP4 outputs (T = 8192, % of the copy bandwidth, stage
  // against row): W = 1, the row kernel ahead at every H = 4096..8192 (by
  // 1.9-18.0 points); W = 2, ahead at H = 8192 (95.1 against 86.1); W = 4,
  // ahead at H <= 5120 (by 3.4-11.4), level at 7168, behind at 8192;
  // W = 8, behind at H >= 5120.
  const bool stage_default =
      auto_long && (quant ? !(W <= 2 || (W < kStageMinW && H <= kRowMaxH))
                          : (W >= kStageMinW && H > kRowMaxH));
  if (vec_ok && pb == 2 && (want == kVariantStage || stage_default) &&
      make_stage_plan(ctx, T, H, &pl, qm == kQuantFp8 ? 1 : (qm == kQuantNvfp4 ? 3 : 0))) {
    *out = pl;
    return FARN_OK;
  }
  if (want == kVariantStage) return FARN_ERR_UNSUPPORTED;
  if (!vec_ok || want == kVariantGeneric) {
    pl.variant = kVariantGeneric;
    pl.cs = 1; pl.vpt = 1; pl.threads = 256;
    pl.grid = T;
  } else {
    int cs = 1;
    if (ctx->force_cluster > 0 && want != kVariantRow) {
      cs = ctx->force_cluster;
    } else if (want != kVariantRow && small &&
               (pb == 2 ? (T < kClusterRowsMax && hv >= 256) : (T < 8 && hv > 512))) {
      // A handful of rows: split each row over a cluster so that every CTA
      // owns about 128 16-byte vectors (bf16 partials) and each thread one
      // vector of every rank, spreading the row's loads over up to 8 SMs.
      // Measured on GB300 (W = 8, H = 4096, back-to-back calls,
      // reduced/residual_out stored after the DSMEM exchange): 4-CTA
      // clusters 1.78 / 1.90 us at T = 1 / 8 against 1.91 / 2.07 us for one
      // CTA per row; at T = 32 and above one CTA per row is faster.  fp32
      // partials keep the earlier rule: rows longer than 4096 elements
      // below 8 rows, about 64 vectors per CTA.
      const int cap = ctx->max_cluster < 8 ? ctx->max_cluster : 8;
      const int64_t min_slice = pb == 2 ? 128 : 64;
      // (The NVFP4 output pairs vectors 2m, 2m+1 inside a CTA: even slices.)
      while (cs * 2 <= cap && hv % (cs * 2) == 0 && hv / (cs * 2) >= min_slice &&
             (qm != kQuantNvfp4 || (hv / (cs * 2)) % 2 == 0))
        cs *= 2;
    }
    if (want == kVariantCluster && cs == 1 && ctx->max_cluster >= 2 && hv % 2 == 0 &&
        (qm != kQuantNvfp4 || hv % 4 == 0))
      cs = 2;
    if (cs > ctx->max_cluster || hv % cs != 0) return FARN_ERR_UNSUPPORTED;
    if (qm == kQuantNvfp4 && (hv / cs) % 2 != 0) return FARN_ERR_UNSUPPORTED;
    const int64_t sv = hv / cs;
    int vpt;
    if (ctx->force_vpt > 0) vpt = ctx->force_vpt;
    else if (small) vpt = sv <= 512 ? 1 : (sv <= 1024 ? 2 : 4);   // loads in one batch
    else vpt = choose_vpt(sv);
    // Many rows of one or two bf16 partials and 256..511 vectors: 4 vectors
    // per thread rather than 2 (GB300, T = 8192, H = 2048: W = 1 / 2 at 93.4
    // / 95.5 % of the copy bandwidth against 84.5 / 91.9 %, with the FP8
    // output 81.4 / 90.2 % against 69.8 / 79.6 %; at W = 4 two stay ahead).
    if (!small && ctx->force_vpt == 0 && pb == 2 && W <= 2 && sv >= 256 && sv < 512) vpt = 4;
    int64_t threads = (sv + vpt - 1) / vpt;
    threads = (threads + 31) / 32 * 32;
    if (threads > 512) {
      // Too long for one CTA's registers: the generic kernel takes it.
      pl.variant = kVariantGeneric;
      pl.cs = 1; pl.vpt = 1; pl.threads = 256; pl.grid = T;
      *out = pl;
      return FARN_OK;
    }
    if (!pick_vec(vpt, cs, pb)) return FARN_ERR_UNSUPPORTED;
    pl.variant = cs > 1 ? kVariantCluster : kVariantRow;
    pl.cs = cs; pl.vpt = vpt; pl.threads = (int)threads;
    pl.grid = T * cs;
    // latency-bound calls of one vector per thread: one CTA (or cluster)
    // per row and no loop (T < small_t, so the grid is small)
    pl.one_row = small && vpt == 1 && pb == 2;
  }
  // Grid limit: rows beyond one pass are looped over inside the kernel.
  const int64_t max_grid = (int64_t)0x7FFFFFFF / pl.cs * pl.cs;
  if (pl.grid > max_grid) pl.grid = max_grid;
  *out = pl;
  return FARN_OK;
}

// The MoE combine's kernel.  Long inputs (T >= the stage threshold) with
// rows longer than 3072 elements (5120 below 8 experts): the TMA-staged
// kernel where a row fits one or two segments of at most 512 consumer
// threads, or more segments of the full 256, else the staged gather kernel,
// which keeps R chunks of gathered rows in flight per thread (GB300,
// T = 4096, K = 8, H = 7168: 98.7 % of the copy bandwidth for the
// TMA-staged kernel, 89.9 % for the staged gather, 81.3 % for one CTA per
// row).  Otherwise one CTA per row, every thread one vector of each
// gathered row for few rows (all loads in flight at once), 4 vectors
// otherwise; the generic kernel for odd shapes and alignments.
// FARN_VARIANT=bulk / stage / row / generic force one of them; FARN_STAGE=0
// leaves long inputs to the row kernel.
int make_moe_plan(const farn_ctx* ctx, int K, int64_t T, int64_t H, bool vec_ok, Plan* out) {
  Plan pl;
  pl.pb = 2; pl.cs = 1; pl.stages = 0; pl.stage_stride = 0; pl.smem = 0; pl.stage_r = 0;
  pl.one_row = false;
  const int64_t hv = H / 8;
  const int want = ctx->force_variant;
  if (want == kVariantCluster) return FARN_ERR_UNSUPPORTED;
  const bool long_moe = long_call(ctx, T, (int64_t)(K + 1) * T * H * 2);
  // Short rows keep the one-CTA-per-row combine kernel even for long calls.
  // Measured on GB300 (T = 4096, % of the copy bandwidth, row / TMA-staged
  // / staged gather): H <= 3072, 69.7-86.2 against 46.1-76.4 / 54.5-64.8
  // (K = 2..16); H = 4096 and 5120 with K <= 6, 82.1-85.3 against
  // 72.8-84.8 / 67.1-79.7.  The TMA-staged kernel also takes rows that need
  // more than two segments when they still get the full 256 consumers
  // (K = 16, H = 8192: 92.0 against 77.8 for the staged gather; K = 8,
  // H = 10240 / 12288: 85.6 / 87.9 against 77.4 / 84.2) but not with fewer
  // (K = 16, H = 7168, 224 consumers: 83.7 against 91.9).
  const bool moe_row = H <= 3072 || (H <= 5120 && K < 8);
  Plan bp;
  if (vec_ok && (want == kVariantBulk ||
                 (want == kVariantAuto && long_moe && (ctx->bulk || (ctx->stage && !moe_row)))) &&
      make_bulk_plan(ctx, K, T, H, &bp, true) &&
      (want == kVariantBulk || ctx->bulk || bp.vpt <= 2 ||
       bp.threads - 32 == farn::kBulkMaxConsumers)) {
    *out = bp;
    return FARN_OK;
  }
  if (want == kVariantBulk) return FARN_ERR_UNSUPPORTED;
  if (vec_ok && want != kVariantGeneric && want != kVariantRow &&
      (want == kVariantStage || (ctx->stage && long_moe && !moe_row)) &&
      make_stage_plan(ctx, T, H, &pl, 2)) {
    *out = pl;
    return FARN_OK;
  }
  if (want == kVariantStage) return FARN_ERR_UNSUPPORTED;
  int vpt = T < ctx->small_t ? (hv <= 512 ? 1 : (hv <= 1024 ? 2 : 4)) : choose_vpt(hv);
  if (ctx->force_vpt > 0) vpt = ctx->force_vpt;
  int64_t threads = ((hv + vpt - 1) / vpt + 31) / 32 * 32;
  if (!vec_ok || threads > 512 || want == kVariantGeneric) {
    pl.variant = kVariantGeneric;
    pl.vpt = 1;
    pl.threads = 256;
  } else {
    pl.variant = kVariantCombine;
    pl.vpt = vpt;
    pl.threads = (int)threads;
  }
  pl.grid = T < 0x7FFFFFFF ? T : 0x7FFFFFFF;
  *out = pl;
  return FARN_OK;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

const char* farn_status_string(int status) {
  switch (status) {
    case FARN_OK: return "ok";
    case FARN_ERR_INVALID_ARG: return "invalid argument";
    case FARN_ERR_UNSUPPORTED: return "unsupported shape or launch configuration";
    case FARN_ERR_ALIAS: return "an output overlaps an input or another output";
    case FARN_ERR_CUDA: return "CUDA runtime error";
    case FARN_ERR_NOMEM: return "out of host memory";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// The argument checks for partials of `pb` bytes per element; with an FP8
// output (qm 1: q_out [T,H] bytes and scale_out [T] floats) or an NVFP4
// output (qm 2: q_out [T,H/2] bytes and scale_out [T,H/16] bytes, H a
// multiple of 16, tensor scale g finite and > 0), both non-null, norm_out
// may be null.
int check_args_pb(const void* const* partials, int W, int pb, const void* residual,
                  const void* weight, float eps, int64_t T, int64_t H,
                  const void* reduced_out, const void* residual_out, const void* norm_out,
                  const void* q_out = nullptr, const void* scale_out = nullptr,
                  int qm = kQuantNone, float g = 1.0f) {
  const bool quant = qm != kQuantNone;
  if (!partials || W < 1 || W > FARN_MAX_W || T < 0 || H < 1) return FARN_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.0f) return FARN_ERR_INVALID_ARG;
  if (qm == kQuantNvfp4 && (H % 16 != 0 || !isfinite(g) || !(g > 0.0f)))
    return FARN_ERR_INVALID_ARG;
  if (H > INT64_MAX / 4 || (T > 0 && T > INT64_MAX / (4 * H))) return FARN_ERR_INVALID_ARG;
  // With no rows nothing is read or written: empty tensors may have null
  // data pointers.
  if (T == 0) return FARN_OK;
  if (!residual || !weight || !reduced_out || !residual_out || (!norm_out && !quant))
    return FARN_ERR_INVALID_ARG;
  if (quant && (!q_out || !scale_out)) return FARN_ERR_INVALID_ARG;
  for (int r = 0; r < W; ++r)
    if (!partials[r]) return FARN_ERR_INVALID_ARG;
  const int64_t nb = T * H * 2, xb = T * H * pb, wb = H * 2;
  // outputs and their byte extents (a null norm_out extends over nothing)
  const void* outs[5] = {reduced_out, residual_out, norm_out, q_out, scale_out};
  const int64_t qb = qm == kQuantFp8 ? T * H : (qm == kQuantNvfp4 ? T * H / 2 : 0);
  const int64_t sb = qm == kQuantFp8 ? T * 4 : (qm == kQuantNvfp4 ? T * H / 16 : 0);
  const int64_t ob[5] = {nb, nb, norm_out ? nb : 0, qb, sb};
  for (int i = 0; i < 5; ++i) {
    for (int j = i + 1; j < 5; ++j)
      if (overlaps(outs[i], ob[i], outs[j], ob[j])) return FARN_ERR_ALIAS;
    for (int r = 0; r < W; ++r)
      if (overlaps(outs[i], ob[i], partials[r], xb)) return FARN_ERR_ALIAS;
    if (overlaps(outs[i], ob[i], weight, wb)) return FARN_ERR_ALIAS;
    const bool inplace_residual = (i == 1 && residual_out == residual);
    if (!inplace_residual && overlaps(outs[i], ob[i], residual, nb)) return FARN_ERR_ALIAS;
  }
  return FARN_OK;
}

int dtype_bytes(int dtype) {
  return dtype == FARN_BF16 ? 2 : (dtype == FARN_F32 ? 4 : 0);
}

}  // namespace

extern "C" {

int farn_check_args(const void* const* partials, int W, const void* residual,
                    const void* weight, float eps, int64_t T, int64_t H,
                    const void* reduced_out, const void* residual_out,
                    const void* norm_out) {
  return check_args_pb(partials, W, 2, residual, weight, eps, T, H, reduced_out, residual_out,
                       norm_out);
}

int farn_create(farn_ctx** out, int device) {
  if (!out || device < 0) return FARN_ERR_INVALID_ARG;
  *out = nullptr;
  // Fault injection for the tests, read here once: "create" fails this
  // call, "launch" makes every launch of the new context fail (before
  // anything is enqueued), "stall" makes CTA 0 of every TMA-staged launch
  // of the new context wait out its time limit (2 s) and report it in the
  // status word.  No per-call environment lookups.
  const char* inject = getenv("FARN_FAULT_INJECT");
  if (inject && strcmp(inject, "create") == 0) return FARN_ERR_CUDA;
  const bool inject_launch = inject && strcmp(inject, "launch") == 0;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) { cudaGetLastError(); return FARN_ERR_CUDA; }
  if (device >= ndev) return FARN_ERR_INVALID_ARG;
  DeviceGuard g(device);
  if (!g.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }

  farn_ctx* c = new (std::nothrow) farn_ctx;
  if (!c) return FARN_ERR_NOMEM;
  c->device = device;
  c->fault_launch = inject_launch ? 1 : 0;
  c->stall_test = inject && strcmp(inject, "stall") == 0 ? 1 : 0;
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete c;
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  // Cluster sizes up to 8 are portable; 16 needs the non-portable opt-in
  // and must still fit on a GPC, which the occupancy query answers.
  c->max_cluster = 8;
  {
    VecKernel k16 = pick_vec(1, 16, 2);
    if (cudaFuncSetAttribute((const void*)k16, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      bool ok16 = true;
      for (int i = 0; i < 8 && ok16; ++i) {
        // the looping kernels (three vector counts, bf16 and fp32
        // partials) and the one-row kernels (with and without the
        // quantised outputs)
        const int vpt = i < 6 ? 1 << (i % 3) : 1, pb = (i >= 3 && i < 6) ? 4 : 2;
        VecKernel k = pick_vec(vpt, 16, pb, i >= 6, i == 6);
        if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) { ok16 = false; break; }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 16; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, (const void*)k, &cfg) != cudaSuccess ||
            nclusters < 1) { ok16 = false; break; }
      }
      if (ok16) c->max_cluster = 16;
    }
    cudaGetLastError();
  }
  c->force_variant = kVariantAuto;
  if (const char* v = getenv("FARN_VARIANT")) {
    if (!strcmp(v, "row")) c->force_variant = kVariantRow;
    else if (!strcmp(v, "cluster")) c->force_variant = kVariantCluster;
    else if (!strcmp(v, "generic")) c->force_variant = kVariantGeneric;
    else if (!strcmp(v, "bulk")) c->force_variant = kVariantBulk;
    else if (!strcmp(v, "stage")) c->force_variant = kVariantStage;
  }
  c->stage = env_int("FARN_STAGE", 1) != 0;
  c->stage_r = env_int("FARN_STAGE_R", 0);
  c->stage_ctas = env_int("FARN_STAGE_CTAS", 0);
  if (c->stage_ctas < 1 || c->stage_ctas > 4) c->stage_ctas = 0;
  c->stage_min_t = env_int("FARN_STAGE_MIN_T", 2048);
  c->stage_min_bytes = (int64_t)env_int("FARN_STAGE_MIN_MB", 128) << 20;
  c->bulk = env_int("FARN_BULK", 0) != 0;
  c->bulk_ctas = env_int("FARN_BULK_CTAS", 1) == 2 ? 2 : 1;
  c->max_smem = 0;
  c->d_status = nullptr;
  if (cudaDeviceGetAttribute(&c->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
      cudaSuccess) {
    delete c;
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  for (int i = 0; i < 10; ++i) {
    if (cudaFuncSetAttribute((const void*)pick_bulk(kBulkVpts[i % 5], i >= 5),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, c->max_smem) !=
        cudaSuccess) {
      delete c;
      cudaGetLastError();
      return FARN_ERR_CUDA;
    }
  }
  memset(c->stage_regs, 0, sizeof c->stage_regs);
  for (int vpt = 2; vpt <= 4; vpt *= 2) {
    for (int i = 0; i < 11; ++i) {
      // dynamic + static shared memory may not exceed the opt-in limit;
      // i < 3: plain kernels, 3..6: FP8-output kernels (depths 16..6),
      // 7..10: NVFP4-output kernels (depths 16..6)
      cudaFuncAttributes fa;
      const int qm = i < 3 ? kQuantNone : (i < 7 ? kQuantFp8 : kQuantNvfp4);
      const int depth = kStageDepths[i < 3 ? i : (i < 7 ? i - 3 : i - 7)];
      const void* k = (const void*)pick_stage(vpt, depth, qm);
      if (cudaFuncGetAttributes(&fa, k) != cudaSuccess ||
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               c->max_smem - (int)fa.sharedSizeBytes) != cudaSuccess) {
        delete c;
        cudaGetLastError();
        return FARN_ERR_CUDA;
      }
      int& regs = c->stage_regs[qm == kQuantNone ? 0 : (qm == kQuantFp8 ? 1 : 3)][vpt >= 4];
      if (fa.numRegs > regs) regs = fa.numRegs;
    }
    for (int i = 0; i < 3; ++i) {       // the staged MoE combine
      cudaFuncAttributes fa;
      const void* k = (const void*)pick_combine_stage(vpt, kStageDepths[i]);
      if (cudaFuncGetAttributes(&fa, k) != cudaSuccess ||
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               c->max_smem - (int)fa.sharedSizeBytes) != cudaSuccess) {
        delete c;
        cudaGetLastError();
        return FARN_ERR_CUDA;
      }
      int& regs = c->stage_regs[2][vpt >= 4];
      if (fa.numRegs > regs) regs = fa.numRegs;
    }
  }
  // The bulk kernel's status word: set on a bounded-wait timeout, read and
  // cleared by farn_device_status.
  if (cudaMalloc((void**)&c->d_status, 256) != cudaSuccess ||
      cudaMemset(c->d_status, 0, 256) != cudaSuccess) {
    if (c->d_status) cudaFree(c->d_status);
    delete c;
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  c->force_cluster = env_int("FARN_CLUSTER", 0);
  if (c->force_cluster != 0 && c->force_cluster != 1 && c->force_cluster != 2 &&
      c->force_cluster != 4 && c->force_cluster != 8 && c->force_cluster != 16)
    c->force_cluster = 0;
  c->pdl = env_int("FARN_PDL", 1) != 0;
  c->small_t = env_int("FARN_SMALL_T", c->num_sms);
  c->force_vpt = env_int("FARN_VPT", 0);
  if (c->force_vpt != 0 && c->force_vpt != 1 && c->force_vpt != 2 && c->force_vpt != 4)
    c->force_vpt = 0;
  *out = c;
  return FARN_OK;
}

int farn_destroy(farn_ctx* ctx) {
  if (ctx) {
    if (ctx->d_status) {
      DeviceGuard g(ctx->device);
      cudaFree(ctx->d_status);
      cudaGetLastError();
    }
    delete ctx;
  }
  return FARN_OK;
}

int farn_device_status(const farn_ctx* ctx, int* status) {
  if (!ctx || !status) return FARN_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }
  int v = 0;
  if (cudaMemcpy(&v, ctx->d_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ctx->d_status, 0, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  *status = v;
  return FARN_OK;
}

static bool vector_path_ok(int W, const void* const* partials, const void* residual,
                           const void* weight, const void* reduced_out,
                           const void* residual_out, const void* norm_out, int64_t H) {
  if (H % 8 != 0) return false;
  for (int r = 0; r < W; ++r)
    if (!aligned16(partials[r])) return false;
  return aligned16(residual) && aligned16(weight) && aligned16(reduced_out) &&
         aligned16(residual_out) && aligned16(norm_out);
}

int farn_plan(const farn_ctx* ctx, int W, int64_t T, int64_t H, const void* const* partials,
              const void* residual, const void* weight, const void* reduced_out,
              const void* residual_out, const void* norm_out, int* variant,
              int* cluster_size, int* threads) {
  return farn_plan_typed(ctx, FARN_BF16, 0, W, T, H, partials, residual, weight, reduced_out,
                         residual_out, norm_out, variant, cluster_size, threads);
}

int farn_plan_typed(const farn_ctx* ctx, int partial_dtype, int flags, int W, int64_t T,
                    int64_t H, const void* const* partials, const void* residual,
                    const void* weight, const void* reduced_out, const void* residual_out,
                    const void* norm_out, int* variant, int* cluster_size, int* threads) {
  if (!ctx || !variant || !cluster_size || !threads) return FARN_ERR_INVALID_ARG;
  const int pb = dtype_bytes(partial_dtype);
  if (!pb || (flags & ~(FARN_PLAN_FP8_OUT | FARN_PLAN_NVFP4_OUT)) ||
      flags == (FARN_PLAN_FP8_OUT | FARN_PLAN_NVFP4_OUT))
    return FARN_ERR_INVALID_ARG;
  const int qm = (flags & FARN_PLAN_FP8_OUT) ? kQuantFp8
                 : (flags & FARN_PLAN_NVFP4_OUT) ? kQuantNvfp4 : kQuantNone;
  const bool quant = qm != kQuantNone;
  if (qm == kQuantNvfp4 && H % 16 != 0) return FARN_ERR_INVALID_ARG;
  // The choice depends on the shape, the dtype, the FP8 flag and the
  // pointers' alignment only; aliasing is not checked here.
  if (!partials || W < 1 || W > FARN_MAX_W || T < 0 || H < 1 || !residual || !weight ||
      !reduced_out || !residual_out || (!norm_out && !quant))
    return FARN_ERR_INVALID_ARG;
  for (int r = 0; r < W; ++r)
    if (!partials[r]) return FARN_ERR_INVALID_ARG;
  Plan pl;
  int st = make_plan(ctx, W, T, H,
                 vector_path_ok(W, partials, residual, weight, reduced_out, residual_out,
                                norm_out ? norm_out : reduced_out, H),
                 pb, &pl, qm, (int64_t)W * T * H * pb + T * H * 2);
  if (st != FARN_OK) return st;
  *variant = pl.variant;
  *cluster_size = pl.cs;
  *threads = pl.threads;
  return FARN_OK;
}

int farn_plan_moe_combine(const farn_ctx* ctx, int K, int64_t T, int64_t H,
                          const void* expert_out, const void* residual, const void* weight,
                          const void* reduced_out, const void* residual_out,
                          const void* norm_out, int* variant, int* threads) {
  if (!ctx || !variant || !threads || K < 1 || K > FARN_MAX_W || T < 0 || H < 1 ||
      !expert_out || !residual || !weight || !reduced_out || !residual_out || !norm_out)
    return FARN_ERR_INVALID_ARG;
  const bool vec_ok = H % 8 == 0 && aligned16(expert_out) && aligned16(residual) &&
                      aligned16(weight) && aligned16(reduced_out) && aligned16(residual_out) &&
                      aligned16(norm_out);
  Plan pl;
  const int st = make_moe_plan(ctx, K, T, H, vec_ok, &pl);
  if (st != FARN_OK) return st;
  *variant = pl.variant;
  *threads = pl.threads;
  return FARN_OK;
}

int farn_forward(const farn_ctx* ctx, const void* const* partials, int W,
                 const void* residual, const void* weight, float eps, int64_t T,
                 int64_t H, void* reduced_out, void* residual_out, void* norm_out,
                 cudaStream_t stream) {
  return farn_forward_typed(ctx, partials, FARN_BF16, W, residual, weight, eps, T, H,
                            reduced_out, residual_out, norm_out, stream);
}

// farn_forward_typed, farn_forward_quant and farn_forward_nvfp4: q_out,
// scale_out, qm and g only for a quantised copy of norm_out (FP8: scale_out
// is float [T]; NVFP4: bytes [T,H/16], g the tensor scale).
static int forward_impl(const farn_ctx* ctx, const void* const* partials, int partial_dtype,
                        int W, const void* residual, const void* weight, float eps, int64_t T,
                        int64_t H, void* reduced_out, void* residual_out, void* norm_out,
                        void* q_out, void* scale_out, int qm, float g, cudaStream_t stream) {
  if (!ctx) return FARN_ERR_INVALID_ARG;
  const int pb = dtype_bytes(partial_dtype);
  if (!pb) return FARN_ERR_INVALID_ARG;
  int st = check_args_pb(partials, W, pb, residual, weight, eps, T, H, reduced_out,
                         residual_out, norm_out, q_out, scale_out, qm, g);
  if (st != FARN_OK) return st;
  if (T == 0) return FARN_OK;
  if (ctx->fault_launch) return FARN_ERR_CUDA;

  Plan pl;
  st = make_plan(ctx, W, T, H,
                 vector_path_ok(W, partials, residual, weight, reduced_out, residual_out,
                                norm_out ? norm_out : reduced_out, H) &&
                     (qm != kQuantFp8 || ((uintptr_t)q_out & 15u) == 0) &&
                     (qm != kQuantNvfp4 || ((uintptr_t)q_out & 3u) == 0),
                 pb, &pl, qm, (int64_t)W * T * H * pb + T * H * 2);
  if (st != FARN_OK) return st;

  farn::Params prm;
  memset(&prm, 0, sizeof prm);
  for (int r = 0; r < W; ++r) prm.x[r] = partials[r];
  prm.residual = residual;
  prm.weight = weight;
  prm.reduced = reduced_out;
  prm.residual_out = residual_out;
  prm.norm_out = norm_out;
  if (qm == kQuantFp8) {
    prm.q_out = static_cast<uint8_t*>(q_out);
    prm.scale_out = static_cast<float*>(scale_out);
  } else if (qm == kQuantNvfp4) {
    prm.fp4_q = static_cast<uint8_t*>(q_out);
    prm.fp4_s = static_cast<uint8_t*>(scale_out);
    prm.fp4_g = g;
  }
  prm.T = T;
  prm.H = H;
  prm.W = W;
  prm.eps = eps;
  prm.err = ctx->d_status;
  prm.stages = pl.stages;
  prm.stage_stride = pl.stage_stride;
  prm.stall_test = ctx->stall_test;
  prm.prefetch = (pl.variant == kVariantRow || pl.variant == kVariantCluster) &&
                 T < ctx->small_t && ctx->pdl;

  DeviceGuard dg(ctx->device);
  if (!dg.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)pl.threads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  // Attributes: the cluster shape of the split-row variant, and
  // programmatic stream serialisation (the kernel waits for the previous
  // grid with griddepcontrol.wait before touching global memory, so this
  // only overlaps launch latency with the previous kernel's tail).
  cudaLaunchAttribute attrs[2];
  unsigned nattr = 0;
  if (pl.cs > 1) {
    attrs[nattr].id = cudaLaunchAttributeClusterDimension;
    attrs[nattr].val.clusterDim.x = (unsigned)pl.cs;
    attrs[nattr].val.clusterDim.y = 1;
    attrs[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  if (ctx->pdl) {
    attrs[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = nattr;

  cudaError_t err;
  if (pl.variant == kVariantGeneric) {
    err = cudaLaunchKernelEx(&cfg, pick_generic(pb), prm);
  } else if (pl.variant == kVariantBulk) {
    err = cudaLaunchKernelEx(&cfg, pick_bulk(pl.vpt), prm);
  } else if (pl.variant == kVariantStage) {
    err = cudaLaunchKernelEx(&cfg, pick_stage(pl.vpt, pl.stage_r, qm), prm);
  } else {
    VecKernel k = pick_vec(pl.vpt, pl.cs, pb, pl.one_row, qm != kQuantNone);
    err = cudaLaunchKernelEx(&cfg, k, prm);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  return FARN_OK;
}

int farn_forward_typed(const farn_ctx* ctx, const void* const* partials, int partial_dtype,
                       int W, const void* residual, const void* weight, float eps, int64_t T,
                       int64_t H, void* reduced_out, void* residual_out, void* norm_out,
                       cudaStream_t stream) {
  return forward_impl(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                      reduced_out, residual_out, norm_out, nullptr, nullptr, kQuantNone, 1.0f,
                      stream);
}

int farn_forward_quant(const farn_ctx* ctx, const void* const* partials, int partial_dtype,
                       int W, const void* residual, const void* weight, float eps, int64_t T,
                       int64_t H, void* reduced_out, void* residual_out, void* norm_out,
                       void* norm_q, float* row_scale, cudaStream_t stream) {
  return forward_impl(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                      reduced_out, residual_out, norm_out, norm_q, row_scale, kQuantFp8, 1.0f,
                      stream);
}

int farn_forward_nvfp4(const farn_ctx* ctx, const void* const* partials, int partial_dtype,
                       int W, const void* residual, const void* weight, float eps, int64_t T,
                       int64_t H, float tensor_scale, void* reduced_out, void* residual_out,
                       void* norm_out, void* norm_fp4, void* block_scale, cudaStream_t stream) {
  return forward_impl(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                      reduced_out, residual_out, norm_out, norm_fp4, block_scale, kQuantNvfp4,
                      tensor_scale, stream);
}

// ------------------------------------------------------------------------
// MoE combine + residual + RMSNorm.
int farn_moe_combine(const farn_ctx* ctx, const void* expert_out, int64_t n_slots,
                     const int32_t* index, const float* gates, int K, const void* residual,
                     const void* weight, float eps, int64_t T, int64_t H, void* reduced_out,
                     void* residual_out, void* norm_out, cudaStream_t stream) {
  if (!ctx || K < 1 || K > FARN_MAX_W || T < 0 || H < 1 || n_slots < 0)
    return FARN_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.0f) return FARN_ERR_INVALID_ARG;
  if (H > INT64_MAX / 4 || (T > 0 && T > INT64_MAX / (4 * H)) ||
      (n_slots > 0 && n_slots > INT64_MAX / (2 * H)))
    return FARN_ERR_INVALID_ARG;
  if (T == 0) return FARN_OK;
  if (!index || !gates || !residual || !weight || !reduced_out || !residual_out || !norm_out ||
      (n_slots > 0 && !expert_out))
    return FARN_ERR_INVALID_ARG;
  if (((uintptr_t)index & 3u) || ((uintptr_t)gates & 3u)) return FARN_ERR_INVALID_ARG;
  const int64_t nb = T * H * 2, eb = n_slots * H * 2, ib = T * K * 4, wb = H * 2;
  const void* outs[3] = {reduced_out, residual_out, norm_out};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], nb, outs[j], nb)) return FARN_ERR_ALIAS;
    if (overlaps(outs[i], nb, expert_out, eb) || overlaps(outs[i], nb, index, ib) ||
        overlaps(outs[i], nb, gates, ib) || overlaps(outs[i], nb, weight, wb))
      return FARN_ERR_ALIAS;
    const bool inplace_residual = (i == 1 && residual_out == residual);
    if (!inplace_residual && overlaps(outs[i], nb, residual, nb)) return FARN_ERR_ALIAS;
  }
  if (ctx->fault_launch) return FARN_ERR_CUDA;

  const bool vec_ok = H % 8 == 0 && aligned16(residual) && aligned16(weight) &&
                      aligned16(reduced_out) && aligned16(residual_out) &&
                      aligned16(norm_out) && (n_slots == 0 || aligned16(expert_out));
  Plan pl;
  const int st = make_moe_plan(ctx, K, T, H, vec_ok, &pl);
  if (st != FARN_OK) return st;
  const bool generic = pl.variant == kVariantGeneric;
  const bool staged = pl.variant == kVariantStage;
  const bool bulk = pl.variant == kVariantBulk;
  farn::Params prm;
  memset(&prm, 0, sizeof prm);
  prm.residual = residual;
  prm.weight = weight;
  prm.reduced = reduced_out;
  prm.residual_out = residual_out;
  prm.norm_out = norm_out;
  prm.T = T;
  prm.H = H;
  prm.W = K;
  prm.eps = eps;
  prm.expert_out = expert_out;
  prm.index = index;
  prm.gates = gates;
  prm.n_slots = n_slots;
  prm.err = ctx->d_status;
  prm.stages = pl.stages;
  prm.stage_stride = pl.stage_stride;
  prm.stall_test = ctx->stall_test;

  DeviceGuard g(ctx->device);
  if (!g.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)pl.threads, 1, 1);
  cfg.dynamicSmemBytes = (staged || bulk) ? pl.smem : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = ctx->pdl ? 1 : 0;
  cudaError_t err;
  if (generic) {
    err = cudaLaunchKernelEx(&cfg, farn::farn_generic_kernel<2, true>, prm);
  } else if (staged) {
    err = cudaLaunchKernelEx(&cfg, pick_combine_stage(pl.vpt, pl.stage_r), prm);
  } else if (bulk) {
    err = cudaLaunchKernelEx(&cfg, pick_bulk(pl.vpt, true), prm);
  } else {
    VecKernel k = pl.vpt == 1 ? &farn::farn_combine_kernel<1>
                  : (pl.vpt == 2 ? &farn::farn_combine_kernel<2> : &farn::farn_combine_kernel<4>);
    err = cudaLaunchKernelEx(&cfg, k, prm);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  return FARN_OK;
}

// ------------------------------------------------------------------------
// No-allocation entry point.
//
// For callers that must not allocate device memory themselves or through
// this library: code that runs inside another framework's plugin or
// allocator interface, where every device allocation has to go through
// that framework, and code that may not call cudaMalloc at all.  It runs
// the TMA-staged kernel (farn_bulk_kernel), whose only memory beyond the
// caller's inputs and outputs is its 4-byte status word; here that word
// lives in the file-scope array below instead of a context's cudaMalloc'd
// block, so nothing is allocated, ever.
//
// The array is kNoAllocScratchBytes (256) bytes per GPU and every GPU that
// loads this library holds it until the process exits.  A call uses its
// first 4 bytes, whatever T, H and W are; the shapes this entry point takes
// are those the TMA-staged kernel's plan takes: 16-byte aligned tensors,
// H % 8 == 0 and H <= 16384 (kBulkMaxH), any W <= 32.
// Others are refused with FARN_ERR_UNSUPPORTED.
//
// The array is shared by every call on the device and keeps the last
// call's contents; each call clears the status word on its stream before
// launching.  Calls that overlap on the GPU (different streams, no
// ordering between them) race on that word.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) int g_farn_noalloc_scratch[kNoAllocScratchBytes / sizeof(int)];

namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  std::mutex mu;
  bool ready = false;           // set-up done (a failed set-up is tried again)
  int* scratch = nullptr;       // device address of g_farn_noalloc_scratch
  int num_sms = 0;
  int max_smem = 0;
};

NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device, with that device current: the scratch array's device
// address (the array's name in host code is only a host-side stand-in),
// the device limits and the bulk kernels' shared-memory attribute.
int noalloc_setup(int device, NoAllocDevice* d) {
  DeviceGuard g(device);
  if (!g.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_farn_noalloc_scratch) != cudaSuccess || !ptr ||
      cudaDeviceGetAttribute(&d->num_sms, cudaDevAttrMultiProcessorCount, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&d->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  for (int vpt : kBulkVpts) {
    if (cudaFuncSetAttribute((const void*)pick_bulk(vpt),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, d->max_smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return FARN_ERR_CUDA;
    }
  }
  d->scratch = static_cast<int*>(ptr);
  return FARN_OK;
}

}  // namespace

int farn_forward_noalloc(int device, const void* const* partials, int W, const void* residual,
                         const void* weight, float eps, int64_t T, int64_t H,
                         void* reduced_out, void* residual_out, void* norm_out,
                         cudaStream_t stream, int* status_out) {
  if (device < 0 || device >= kNoAllocMaxDevices) return FARN_ERR_INVALID_ARG;
  int st = farn_check_args(partials, W, residual, weight, eps, T, H, reduced_out,
                           residual_out, norm_out);
  if (st != FARN_OK) return st;
  if (T == 0) {
    if (status_out) *status_out = 0;
    return FARN_OK;
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) { cudaGetLastError(); return FARN_ERR_CUDA; }
  if (device >= ndev) return FARN_ERR_INVALID_ARG;
  NoAllocDevice* d = &g_noalloc_dev[device];
  {
    std::lock_guard<std::mutex> lock(d->mu);
    if (!d->ready) {
      st = noalloc_setup(device, d);
      if (st != FARN_OK) return st;
      d->ready = true;
    }
  }
  static_assert(sizeof(int) <= kNoAllocScratchBytes, "status word must fit the scratch array");

  if (!vector_path_ok(W, partials, residual, weight, reduced_out, residual_out, norm_out, H))
    return FARN_ERR_UNSUPPORTED;
  // The plan of the TMA-staged kernel for this device: a context-shaped
  // description of the device on the stack (no device memory behind it).
  farn_ctx dc;
  memset(&dc, 0, sizeof dc);
  dc.device = device;
  dc.num_sms = d->num_sms;
  dc.max_smem = d->max_smem;
  dc.bulk_ctas = 1;
  dc.force_variant = kVariantBulk;
  Plan pl;
  if (!make_bulk_plan(&dc, W, T, H, &pl)) return FARN_ERR_UNSUPPORTED;

  farn::Params prm;
  memset(&prm, 0, sizeof prm);
  for (int r = 0; r < W; ++r) prm.x[r] = partials[r];
  prm.residual = residual;
  prm.weight = weight;
  prm.reduced = reduced_out;
  prm.residual_out = residual_out;
  prm.norm_out = norm_out;
  prm.T = T;
  prm.H = H;
  prm.W = W;
  prm.eps = eps;
  prm.err = d->scratch;
  prm.stages = pl.stages;
  prm.stage_stride = pl.stage_stride;

  DeviceGuard g(device);
  if (!g.ok) { cudaGetLastError(); return FARN_ERR_CUDA; }
  if (cudaMemsetAsync(d->scratch, 0, sizeof(int), stream) != cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)pl.threads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, pick_bulk(pl.vpt), prm) != cudaSuccess) {
    cudaGetLastError();
    return FARN_ERR_CUDA;
  }
  if (status_out) {
    int v = 0;
    if (cudaMemcpyAsync(&v, d->scratch, sizeof v, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
      cudaGetLastError();
      return FARN_ERR_CUDA;
    }
    *status_out = v;
  }
  return FARN_OK;
}

}  // extern "C"
