// Device code of the fused rank-sum + residual add + RMSNorm operator for
// sm_103a (GB300).
//
// Operation: FlagTree pull request "[TLERaw] Add NVSHMEM allreduce RMSNorm
// tutorial", Summary (reduced = sum of the rank partials, residual_out =
// reduced + residual, norm_out = RMSNorm(residual_out, weight, eps)) and
// Implementation section 3 (the residual + RMSNorm epilogue with FP32
// accumulation), fused into one pass over HBM.
//
// The page maps one token row to one CTA (Implementation section 2).  That
// mapping is kept for most calls (farn_vec_kernel with CS == 1).  For a
// handful of rows, where one CTA per row would leave most of the 152 SMs
// idle, a thread-block cluster of CS CTAs splits each row; the CTAs of a
// cluster exchange their partial sums of squares through distributed
// shared memory (DSMEM).  Long inputs of many partials, or with the
// quantised outputs, take persistent kernels that stage the rows in shared
// memory (farn_stage_kernel with cp.async, farn_bulk_kernel with TMA bulk
// copies).
//
// Per element the arithmetic is fixed (f = exact bf16 -> fp32 widening,
// bf16 = round to nearest even):
//   acc = -0.0f; for r in 0..W-1: acc += f(x[r])      // -0 is the exact
//   red = bf16(acc)                                    // additive identity,
//   ro  = bf16(f(red) + f(residual))                   // so acc == f(x[0])
//   ss += f(ro)^2                                      // after rank 0
//   norm = bf16((f(ro) * rstd) * f(weight)),  rstd = 1/sqrt(ss/H + eps)
// so `reduced` and `residual_out` do not depend on the launch shape; only
// the order of the row's sum of squares does.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace farn {

constexpr int kMaxW = 32;

// Kernel parameters, passed by value (__grid_constant__): the W partial
// pointers are indexed by rank straight from the parameter bank.
struct Params {
  const void* x[kMaxW];
  const void* residual;
  const void* weight;
  void* reduced;
  void* residual_out;
  void* norm_out;
  int64_t T;     // rows
  int64_t H;     // elements per row
  int W;         // partials
  float eps;
  // optional FP8 (E4M3) output of norm_out, row kernels only: q_out [T,H]
  // bytes and scale_out [T] fp32, or null; norm_out may then be null too
  uint8_t* q_out;
  float* scale_out;
  // optional NVFP4 output of norm_out (row, cluster, generic and stage
  // kernels): fp4_q [T,H/2] bytes of E2M1 codes (element 2i in the low
  // nibble), fp4_s [T,H/16] E4M3 block scales, fp4_g the tensor scale;
  // H % 16 == 0.  Null when not wanted.
  uint8_t* fp4_q;
  uint8_t* fp4_s;
  float fp4_g;
  // row and cluster kernels: prefetch each CTA's first row into L2 before
  // waiting for the previous kernel (set for latency-bound calls)
  int prefetch;
  // MoE combine only (farn_combine_kernel, farn_generic_kernel<2, true>):
  // W is K, the experts per token
  const void* expert_out;  // bf16 [n_slots, H]
  const int32_t* index;    // [T, K]; -1 or out of [0, n_slots): skipped
  const float* gates;      // [T, K]
  int64_t n_slots;
  // bulk (TMA-staged) kernel only
  int* err;               // device status word, bits of kBulkErr* on a timeout
  uint32_t stages;        // shared-memory ring stages
  uint32_t stage_stride;  // bytes per input slot of a stage (multiple of 128)
  // a test of the bounded waits: CTA 0's consumers wait on a barrier that
  // nothing completes, give up after the time limit and abort the CTA
  int stall_test;
};

// ----------------------------------------------------------- bf16 helpers
// The two bf16 values of a 32-bit word: element 2e is the low half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two fp32 values to bf16 (nearest even) and pack them, lo in the
// low half.  One cvt.rn.bf16x2.f32 instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t to_bf16(float v) {
  return (uint16_t)(pack_bf16x2(v, 0.0f) & 0xFFFFu);
}

// Two fp32 values to E4M3 (round to nearest even, finite saturation),
// lo in the low byte.  One cvt.rn.satfinite.e4m3x2.f32.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// The per-row FP8 scale written for dequantisation, amax / 448, and the
// inverse the values are multiplied by, 448 / amax (each one IEEE fp32
// division per row; both 1 for an all-zero row).
__device__ __forceinline__ float e4m3_row_scale(float amax) {
  return amax > 0.0f ? amax / 448.0f : 1.0f;
}
__device__ __forceinline__ float e4m3_row_inv(float amax) {
  return amax > 0.0f ? 448.0f / amax : 1.0f;
}

// Two fp32 values to E2M1 (round to nearest even, finite saturation), lo in
// bits 0-3 and hi in bits 4-7.  One cvt.rn.satfinite.e2m1x2.f32.
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The value of an E4M3 byte (exact: E4M3 -> f16 -> f32).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .b32 x;\n\tcvt.rn.f16x2.e4m3x2 x, %1;\n\t"
      "mov.b32 {lo, hi}, x;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "h"((uint16_t)b));
  return f;
}

// NVFP4 codes of one 16-byte vector nv (8 bf16 values of norm_out) whose
// 16-element block is completed by the vector of lane ^ 1; every lane of
// the warp calls it.  Block amax (NaN ignored) -> E4M3 scale
// s = E4M3((amax / 6) * g) -> inv = g / value(s) (IEEE divisions) ->
// E2M1(x * inv) with magnitudes above 6 saturated (min(x, 6) also sends a
// NaN to +6); a block whose scale is 0 gets all-zero codes.  Returns the 8
// codes (element 2i in the low nibble of byte i); *sb gets the scale byte.
__device__ __forceinline__ uint32_t nvfp4_vec(uint4 nv, float g, uint32_t* sb) {
  const uint32_t n[4] = {nv.x, nv.y, nv.z, nv.w};
  float mx = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fmaxf(fabsf(bf_lo(n[e])), fabsf(bf_hi(n[e]))));
  mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  const uint32_t s = pack_e4m3x2((mx / 6.0f) * g, 0.0f) & 0xFFu;
  const float sv = e4m3_to_f32(s);
  const float inv = g / sv;
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    word |= pack_e2m1x2(fminf(bf_lo(n[e]) * inv, 6.0f), fminf(bf_hi(n[e]) * inv, 6.0f))
            << (8 * e);
  *sb = s;
  return sv > 0.0f ? word : 0u;
}

__device__ __forceinline__ void st_stream_u32(uint8_t* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// ----------------------------------------------------------- memory access
// Partials: read once, never written by this kernel -> non-coherent path,
// no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Residual: coherent load (residual_out may be the same buffer; every
// element is read before the same thread overwrites it).
__device__ __forceinline__ uint4 ld_coherent(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Weight: shared by every row, keep it cached.
__device__ __forceinline__ uint4 ld_keep(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Outputs: written once, streamed out (evict-first).
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Eight fp32 partial values (two 16-byte vectors) added in place.
__device__ __forceinline__ void add8f(float* acc, uint4 a, uint4 b) {
  acc[0] += __uint_as_float(a.x); acc[1] += __uint_as_float(a.y);
  acc[2] += __uint_as_float(a.z); acc[3] += __uint_as_float(a.w);
  acc[4] += __uint_as_float(b.x); acc[5] += __uint_as_float(b.y);
  acc[6] += __uint_as_float(b.z); acc[7] += __uint_as_float(b.w);
}

// Eight bf16 values (one 16-byte vector) added in place.  The mixed-precision
// add.rn.f32.bf16 widens its bf16 operand (exactly) and rounds the fp32 sum
// once: the same addition as acc + bf_lo/bf_hi(v), one instruction per
// element instead of an unpack and an add.
__device__ __forceinline__ void add8(float* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(acc[2 * e]), "+f"(acc[2 * e + 1]) : "r"(w[e]));
}

// The same eight additions two at a time: the halves of each 32-bit word
// unpacked and added with one packed add.rn.f32x2 (each lane an IEEE fp32
// addition, so the sums are those of add8).  Measured on GB300, the plain
// stage kernel streams faster with this form (nonpow2 99.8 % vs 89 % of
// the copy bandwidth, prefill 103.6 % vs 99.4 %), the quantising stage
// kernels, the TMA-staged kernel and the latency-bound row kernels with
// add8 (FP8 94.6 % vs 91.5 %, NVFP4 92.3 % vs 90.3 %, bulk at nonpow2
// 98.9 % vs 94.3 %).
__device__ __forceinline__ void add8_x2(float* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint64_t a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc[2 * e]), "f"(acc[2 * e + 1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "r"(w[e] << 16), "r"(w[e] & 0xFFFF0000u));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2 * e]), "=f"(acc[2 * e + 1]) : "l"(a));
  }
}

// acc[0..8) += g * f(v) for the eight bf16 values of one 16-byte vector,
// the product and the sum each rounded to fp32 (__fmul_rn / __fadd_rn are
// never fused into a multiply-add).  A packed form, mul.rn.f32x2 followed
// by add.rn.f32x2 (explicit rounding on both), did not keep the products
// separately rounded inside the combine kernels with this toolchain: on
// GB300 the reduced values of a 32-expert call (T = 700, H = 1024) equal
// those of a fused multiply-add in every one of 716,800 elements and differ
// from the separately rounded sums in 48, built with or without
// -fmad=false (an isolated kernel doing the same pair kept them separate).
// It was no faster either (the staged combine at 88.3 % of the copy
// bandwidth both ways), nor were scalar products with packed sums.
__device__ __forceinline__ void gate_add8(float* acc, float g, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(g, bf_lo(w[e])));
    acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(g, bf_hi(w[e])));
  }
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Write a float into the shared memory of CTA `rank` of this cluster, at
// the address that `local` has in this CTA.
__device__ __forceinline__ void st_dsmem_f32(float* local, uint32_t rank, float v) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(remote), "f"(v) : "memory");
}

// ------------------------------------------- programmatic dependent launch
// When launched with programmatic stream serialisation the grid may start
// while the previous kernel on the stream is still finishing.  pdl_wait()
// blocks until that kernel has completed and its memory is visible, so no
// global load or store may come before it.  pdl_trigger() lets the next
// kernel start launching.  Both are no-ops for an ordinary launch.
// A hint that pulls the 128-byte line at p into L2.  It changes nothing a
// later load observes (the PTX memory model gives prefetches no effect on
// ordering or values, and L2 is where every write lands), so it may run
// before griddepcontrol.wait.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// The CTA total (maximum) of the per-warp partials ws[0..nw), nw <= 32,
// formed by every warp at once: one shared-memory load per lane and a
// butterfly.  Every lane of every warp gets the same bits (IEEE addition
// and max are commutative and all lanes combine the same pairs), and the
// serial chain of nw dependent loads and adds is gone.  Full warps only.
__device__ __forceinline__ float sum_partials(const float* ws, int nw, int lane) {
  return warp_sum(lane < nw ? ws[lane] : 0.0f);
}
__device__ __forceinline__ float max_partials(const float* wm, int nw, int lane) {
  return warp_max(lane < nw ? wm[lane] : 0.0f);
}

// --------------------------------------------------------- vector kernel
// Each CTA owns the column slice `slice` (of CS) of one row; each thread
// owns VPT 16-byte vectors (8 bf16 each) of that slice, at
// j = threadIdx.x + k*blockDim.x.  The slice is sv = H/8/CS vectors; the
// host guarantees H % 8 == 0, (H/8) % CS == 0, 16-byte aligned pointers and
// blockDim.x * VPT >= sv.
//
// Partials are loaded G ranks at a time (G*VPT*PV = 8 16-byte loads in
// flight per thread per batch, plus the residual) and added in rank order.
// PB is the partials' element size: 2 (bf16) or 4 (fp32, two 16-byte loads
// per 8 elements); residual, weight and outputs are bf16 either way.  At
// most 512 threads per CTA (128 registers per thread); the one-vector bf16
// one-row and single-CTA instantiations are built for two CTAs of 512
// threads per SM (64 registers), so that the next call's CTAs can start on
// an SM while this call's CTA still runs there.  ONE_ROW (latency-bound calls, one CTA or
// cluster per row, grid = T * CS): no loop over rows, which leaves the
// registers to fetch the weight together with the partials.  QUANT: the
// FP8 / NVFP4 outputs are compiled in; the one-row builds of plain calls
// leave them out, which shortens their code (GB300, W = 8, H = 4096,
// back-to-back calls: T = 1 / 8 / 64 at 1.98 / 2.14 / 2.41 us against
// 2.03 / 2.19 / 2.44 us with them in).
template <int VPT, int CS, int PB = 2, bool ONE_ROW = false, bool QUANT = true>
__global__ void __launch_bounds__(512, (VPT == 1 && PB == 2 && (ONE_ROW || CS == 1)) ? 2 : 1)
farn_vec_kernel(const __grid_constant__ Params p) {
  constexpr int PV = PB / 2;
  constexpr int G = (8 / (VPT * PV)) > 0 ? (8 / (VPT * PV)) : 1;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  const int64_t hv = p.H >> 3;
  const int sv = (int)(hv / CS);
  const uint32_t slice = (CS == 1) ? 0u : cluster_ctarank();
  const float Hf = (float)p.H;

  __shared__ float warp_ss[2][32];
  __shared__ float cluster_ss[2][CS];   // [row parity][CTA rank in cluster]
  __shared__ float warp_mx[2][32];      // FP8 output only: row amax
  __shared__ float cluster_mx[2][CS];

  const uint4* __restrict__ wv4 = reinterpret_cast<const uint4*>(p.weight) + (int64_t)slice * sv;
  // One-row calls and two vectors per thread: the weight is fetched with
  // the first batch of partials (latency-bound calls).  Otherwise it is
  // fetched after the rank loop, where it holds no registers during the
  // loads and its latency hides behind the row reduction (the looping
  // one-vector build then fits 64 registers with no spill).
  constexpr bool kEarlyWeight = VPT == 2 || ONE_ROW;
  uint4 wv[VPT];

  // Latency-bound calls (the host sets p.prefetch when there are fewer rows
  // than SMs): while the previous kernel on the stream finishes
  // (programmatic dependent launch), pull this CTA's first row of every
  // input into L2, one prefetch per 128-byte line, so the loads after
  // griddepcontrol.wait find it there instead of paying a DRAM round trip.
  // The loads still observe everything the previous kernel wrote.  (Long
  // inputs skip it: there every CTA's first row is its only row and the
  // extra requests cost bandwidth, 102.6 % -> 92.2 % with fp32 partials.)
  if (p.prefetch) {
    const int64_t row0 = blockIdx.x / CS;
    if (row0 < p.T) {
      const int64_t b0 = row0 * hv + (int64_t)slice * sv;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        if (j < sv && ((j * PV) & 7) == 0) {
          for (int r = 0; r < p.W; ++r)
            prefetch_l2(reinterpret_cast<const uint4*>(p.x[r]) + (b0 + j) * PV);
        }
        if (j < sv && (j & 7) == 0) {
          prefetch_l2(reinterpret_cast<const uint4*>(p.residual) + b0 + j);
          prefetch_l2(wv4 + j);
        }
      }
    }
  }

  pdl_wait();
  // Latency-bound calls let the next kernel on the stream start launching
  // as soon as this one is released: its CTAs then prefetch their rows into
  // L2 during the whole of this call, one call ahead and no further (that
  // kernel releases the one after it only once this one has finished).
  // Measured on GB300 (W = 8, H = 4096, back-to-back calls): T = 64 from
  // 2.62 to 2.28 us with two CTAs per SM, T = 128 from 3.35 to 2.87 us;
  // triggering before the wait instead lets launches run many calls ahead
  // and was slower (T = 64: 3.26 us).
  if (p.prefetch) pdl_trigger();

  const int64_t rows_per_pass = gridDim.x / CS;
  int it = 0;
  for (int64_t row = blockIdx.x / CS; row < p.T;
       row = ONE_ROW ? p.T : row + rows_per_pass, ++it) {
    const int64_t base = row * hv + (int64_t)slice * sv;   // vector offset

    uint4 rv[VPT];
    float acc[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] = -0.0f;

    // a1: rank sum in fp32, rank order 0..W-1, G ranks per batch of loads.
    // The first batch names its partials by constant rank indices (x[g]
    // straight from the parameter bank) and is issued before the residual
    // and weight loads, which come before its adds; later batches index the
    // pointer array at run time.  Measured on GB300 (W = 8, H = 4096,
    // back-to-back calls, T = 64): 2.86 us with every batch indexed at run
    // time, 2.45 us with the first batch constant and the residual loaded
    // first, 2.34 us in this order.
    auto load_batch = [&](int r0, bool constant_index, uint4 (&xv)[G][VPT][PV]) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int r = r0 + g;
        const uint4* xp = reinterpret_cast<const uint4*>(
                              constant_index ? p.x[g] : p.x[r < p.W ? r : 0]) + base * PV;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int j = tid + k * blockDim.x;
#pragma unroll
          for (int v = 0; v < PV; ++v) {
            xv[g][k][v] = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.W && j < sv) xv[g][k][v] = ld_stream(xp + j * PV + v);
          }
        }
      }
    };
    auto add_batch = [&](int r0, const uint4 (&xv)[G][VPT][PV]) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (r0 + g < p.W) {
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            if (PB == 2) add8(acc[k], xv[g][k][0]);
            else add8f(acc[k], xv[g][k][0], xv[g][k][PV - 1]);
          }
        }
      }
    };
    {
      uint4 xv[G][VPT][PV];
      load_batch(0, true, xv);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        if (j < sv) {
          rv[k] = ld_coherent(reinterpret_cast<const uint4*>(p.residual) + base + j);
          if (kEarlyWeight) wv[k] = ld_keep(wv4 + j);
        }
      }
      add_batch(0, xv);
    }
    for (int r0 = G; r0 < p.W; r0 += G) {
      uint4 xv[G][VPT][PV];
      load_batch(r0, false, xv);
      add_batch(r0, xv);
    }

    // a2 + a5: reduced and residual_out, rounded and stored; a3: the
    // thread's part of the sum of squares of the rounded residual_out.
    // In a one-row cluster the two stores wait until after the DSMEM
    // exchange below: its release would otherwise wait for them to reach
    // memory (measured on GB300, 4-CTA clusters at T = 1..8, H = 4096:
    // about 0.3 us per call).
    constexpr bool kLateStores = CS > 1 && ONE_ROW;
    uint4 ro[VPT], rd[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * blockDim.x;
      if (j < sv) {
        const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        uint32_t red[4], out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          red[e] = pack_bf16x2(acc[k][2 * e], acc[k][2 * e + 1]);
          const float s0 = bf_lo(red[e]) + bf_lo(rw[e]);
          const float s1 = bf_hi(red[e]) + bf_hi(rw[e]);
          out[e] = pack_bf16x2(s0, s1);
          const float q0 = bf_lo(out[e]), q1 = bf_hi(out[e]);
          ss = fmaf(q0, q0, ss);
          ss = fmaf(q1, q1, ss);
        }
        rd[k] = make_uint4(red[0], red[1], red[2], red[3]);
        ro[k] = make_uint4(out[0], out[1], out[2], out[3]);
        if (!kLateStores) {
          st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j, rd[k]);
          st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
        }
      }
    }

    // Last loads of this row issued: the next kernel may start launching.
    if (row + rows_per_pass >= p.T) pdl_trigger();

    // The weight slice (cached: every row reads it) is fetched here for
    // large slices, so its latency hides behind the reduction below.
    if (!kEarlyWeight) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        if (j < sv) wv[k] = ld_keep(wv4 + j);
      }
    }

    // a3: CTA sum of squares (warp butterfly, then a butterfly over the
    // warps' sums in every warp; every thread forms the same total).
    ss = warp_sum(ss);
    float* ws = warp_ss[it & 1];
    if (lane == 0) ws[warp] = ss;
    __syncthreads();
    float tot = sum_partials(ws, nwarps, lane);

    if (CS > 1) {
      // Cluster: thread c pushes this CTA's total into slot [slice] of CTA
      // c through DSMEM; one cluster barrier (release/acquire) later every
      // CTA holds all CS totals in its own shared memory and sums them in
      // CTA-rank order, so all CTAs of the row get the same rstd.  No
      // remote access follows the barrier, so a CTA may exit right after
      // it; the row-parity double buffer keeps the next row's pushes off
      // slots a slower peer is still reading.
      float* slots = cluster_ss[it & 1];
      if (tid < CS) st_dsmem_f32(&slots[slice], (uint32_t)tid, tot);
      cluster_arrive_release();
      cluster_wait_acquire();
      tot = 0.0f;
#pragma unroll
      for (int c = 0; c < CS; ++c) tot += slots[c];
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        if (kLateStores && j < sv) {
          st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j, rd[k]);
          st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
        }
      }
    }

    // a4: rstd with IEEE division and square root, then the normalised,
    // weighted output.
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
    uint4 nb[VPT];
    float mx = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * blockDim.x;
      nb[k] = make_uint4(0u, 0u, 0u, 0u);
      if (j < sv) {
        const uint32_t q[4] = {ro[k].x, ro[k].y, ro[k].z, ro[k].w};
        const uint32_t w[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
        uint32_t n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n0 = (bf_lo(q[e]) * rstd) * bf_lo(w[e]);
          const float n1 = (bf_hi(q[e]) * rstd) * bf_hi(w[e]);
          n[e] = pack_bf16x2(n0, n1);
        }
        nb[k] = make_uint4(n[0], n[1], n[2], n[3]);
        if (p.norm_out) st_stream(reinterpret_cast<uint4*>(p.norm_out) + base + j, nb[k]);
      }
    }

    if (QUANT && p.q_out) {
      // FP8 output: the row's amax of the bf16 norm_out (fmaxf ignores NaN;
      // max is exact, so every CTA and thread gets the same value), then
      // E4M3(norm_out * (448 / amax)) for each element.
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const uint32_t n[4] = {nb[k].x, nb[k].y, nb[k].z, nb[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(bf_lo(n[e])), fabsf(bf_hi(n[e]))));
      }
      mx = warp_max(mx);
      float* wm = warp_mx[it & 1];
      if (lane == 0) wm[warp] = mx;
      __syncthreads();
      float amax = max_partials(wm, nwarps, lane);
      if (CS > 1) {
        float* slots = cluster_mx[it & 1];
        if (tid < CS) st_dsmem_f32(&slots[slice], (uint32_t)tid, amax);
        cluster_arrive_release();
        cluster_wait_acquire();
        for (int c = 0; c < CS; ++c) amax = fmaxf(amax, slots[c]);
      }
      const float scale = e4m3_row_scale(amax);
      const float inv = e4m3_row_inv(amax);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        if (j < sv) {
          const uint32_t n[4] = {nb[k].x, nb[k].y, nb[k].z, nb[k].w};
          uint32_t q8[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            q8[e] = pack_e4m3x2(bf_lo(n[e]) * inv, bf_hi(n[e]) * inv);
          const uint2 out = make_uint2(q8[0] | (q8[1] << 16), q8[2] | (q8[3] << 16));
          asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};"
                       :: "l"(p.q_out + (base + j) * 8), "r"(out.x), "r"(out.y) : "memory");
        }
      }
      if (tid == 0 && slice == 0) p.scale_out[row] = scale;
    }

    if (QUANT && p.fp4_q) {
      // NVFP4 output: blocks of 16 elements are vector pairs (j, j ^ 1) of
      // neighbouring lanes (the host keeps the slice's vector count even).
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * blockDim.x;
        uint32_t sb;
        const uint32_t codes = nvfp4_vec(nb[k], p.fp4_g, &sb);
        if (j < sv) {
          st_stream_u32(p.fp4_q + (base + j) * 4, codes);
          if ((j & 1) == 0) p.fp4_s[(base + j) >> 1] = (uint8_t)sb;
        }
      }
    }
  }
}

// -------------------------------------------------------- generic kernel
// Any H, any alignment: one CTA per row, scalar bf16 accesses, two passes
// (the second re-reads the residual_out this same thread wrote).
template <int PB = 2, bool COMBINE = false>
__global__ void __launch_bounds__(256)
farn_generic_kernel(const __grid_constant__ Params p) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  const float Hf = (float)p.H;
  __shared__ float warp_ss[2][32];
  const uint16_t* res = reinterpret_cast<const uint16_t*>(p.residual);
  const uint16_t* wt = reinterpret_cast<const uint16_t*>(p.weight);
  uint16_t* red_out = reinterpret_cast<uint16_t*>(p.reduced);
  uint16_t* ro_out = reinterpret_cast<uint16_t*>(p.residual_out);
  uint16_t* nrm_out = reinterpret_cast<uint16_t*>(p.norm_out);
  pdl_wait();
  int it = 0;
  for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x, ++it) {
    const int64_t off = row * p.H;
    float ss = 0.0f;
    for (int64_t h = tid; h < p.H; h += blockDim.x) {
      float acc = -0.0f;
      if constexpr (COMBINE) {
        // MoE combine: gates * gathered expert rows, product and sum each
        // rounded (no fused multiply-add), k in order, bad slots skipped
        const uint16_t* ex = reinterpret_cast<const uint16_t*>(p.expert_out);
        for (int k = 0; k < p.W; ++k) {
          const int32_t sl = p.index[row * p.W + k];
          if (sl < 0 || (int64_t)sl >= p.n_slots) continue;
          const float x = __uint_as_float((uint32_t)ex[(int64_t)sl * p.H + h] << 16);
          acc = __fadd_rn(acc, __fmul_rn(p.gates[row * p.W + k], x));
        }
      } else {
        for (int r = 0; r < p.W; ++r) {
          if (PB == 2)
            acc += __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(p.x[r])[off + h] << 16);
          else
            acc += reinterpret_cast<const float*>(p.x[r])[off + h];
        }
      }
      const uint16_t rb = to_bf16(acc);
      red_out[off + h] = rb;
      const float s = __uint_as_float((uint32_t)rb << 16) +
                      __uint_as_float((uint32_t)res[off + h] << 16);
      const uint16_t ob = to_bf16(s);
      ro_out[off + h] = ob;
      const float q = __uint_as_float((uint32_t)ob << 16);
      ss = fmaf(q, q, ss);
    }
    ss = warp_sum(ss);
    float* ws = warp_ss[it & 1];
    if (lane == 0) ws[warp] = ss;
    __syncthreads();
    float tot = sum_partials(ws, nwarps, lane);
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
    float mx = 0.0f;
    for (int64_t h = tid; h < p.H; h += blockDim.x) {
      const float q = __uint_as_float((uint32_t)ro_out[off + h] << 16);
      const float w = __uint_as_float((uint32_t)wt[h] << 16);
      const uint16_t nbits = to_bf16((q * rstd) * w);
      if (nrm_out) nrm_out[off + h] = nbits;
      mx = fmaxf(mx, fabsf(__uint_as_float((uint32_t)nbits << 16)));
    }
    if (p.q_out) {
      // FP8 output: row amax, then a third pass that recomputes each
      // normalised value (same arithmetic, same bits) and quantises it.
      __shared__ float warp_mx[2][32];
      mx = warp_max(mx);
      float* wm = warp_mx[it & 1];
      if (lane == 0) wm[warp] = mx;
      __syncthreads();
      float amax = max_partials(wm, nwarps, lane);
      const float scale = e4m3_row_scale(amax);
      const float inv = e4m3_row_inv(amax);
      for (int64_t h = tid; h < p.H; h += blockDim.x) {
        const float q = __uint_as_float((uint32_t)ro_out[off + h] << 16);
        const float w = __uint_as_float((uint32_t)wt[h] << 16);
        const float n = __uint_as_float((uint32_t)to_bf16((q * rstd) * w) << 16);
        p.q_out[off + h] = (uint8_t)(pack_e4m3x2(n * inv, 0.0f) & 0xFFu);
      }
      if (tid == 0) p.scale_out[row] = scale;
    }
    if (p.fp4_q) {
      // NVFP4 output: a third pass, every lane on every step so that the
      // 16 lanes of a block (blockDim.x is a multiple of 16, H % 16 == 0)
      // reduce its amax and pair their codes by shuffles.
      for (int64_t h0 = 0; h0 < p.H; h0 += blockDim.x) {
        const int64_t h = h0 + tid;
        const bool in = h < p.H;
        float n = 0.0f;
        if (in) {
          const float q = __uint_as_float((uint32_t)ro_out[off + h] << 16);
          const float w = __uint_as_float((uint32_t)wt[h] << 16);
          n = __uint_as_float((uint32_t)to_bf16((q * rstd) * w) << 16);
        }
        float bmx = fmaxf(0.0f, fabsf(n));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) bmx = fmaxf(bmx, __shfl_xor_sync(0xFFFFFFFFu, bmx, o));
        const uint32_t s = pack_e4m3x2((bmx / 6.0f) * p.fp4_g, 0.0f) & 0xFFu;
        const float sv = e4m3_to_f32(s);
        const float inv = p.fp4_g / sv;
        uint32_t code = pack_e2m1x2(fminf(n * inv, 6.0f), 0.0f) & 0xFu;
        if (!(sv > 0.0f)) code = 0;
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, code, 1);
        if (in && (h & 1) == 0) p.fp4_q[(off + h) >> 1] = (uint8_t)(code | (other << 4));
        if (in && (h & 15) == 0) p.fp4_s[(off + h) >> 4] = (uint8_t)s;
      }
    }
  }
}

// ------------------------------------------------------ MoE combine kernel
// The per-token weighted sum of its K expert rows (the MoE "local y
// reduce"), fused with the same residual add + RMSNorm epilogue as
// farn_vec_kernel (one CTA per row).  Row t reads index[t,0..K) and
// gates[t,0..K) (every thread the same K words: broadcast through L1), then
// gathers 16-byte vectors of the selected rows of expert_out, G slots at a
// time, and accumulates gate * x with the product and the sum each rounded
// to fp32 (gate_add8: no fused multiply-add), k in order.
// Slots outside [0, n_slots) are skipped, so a bad index never leads to an
// out-of-bounds load.
template <int VPT>
__global__ void __launch_bounds__(512)
farn_combine_kernel(const __grid_constant__ Params p) {
  constexpr int G = (8 / VPT) > 0 ? (8 / VPT) : 1;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  const int64_t hv = p.H >> 3;
  const int sv = (int)hv;
  const int K = p.W;
  const float Hf = (float)p.H;
  __shared__ float warp_ss[2][32];
  const uint4* __restrict__ wv4 = reinterpret_cast<const uint4*>(p.weight);
  const uint4* __restrict__ ex4 = reinterpret_cast<const uint4*>(p.expert_out);

  pdl_wait();
  int it = 0;
  for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x, ++it) {
    const int64_t base = row * hv;
    uint4 rv[VPT];
    float acc[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * blockDim.x;
      if (j < sv) rv[k] = ld_coherent(reinterpret_cast<const uint4*>(p.residual) + base + j);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] = -0.0f;
    }
    for (int k0 = 0; k0 < K; k0 += G) {
      uint4 xv[G][VPT];
      float gt[G];
      bool ok[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int k = k0 + g;
        int32_t sl = -1;
        gt[g] = 0.0f;
        if (k < K) {
          sl = __ldg(p.index + row * K + k);
          gt[g] = __ldg(p.gates + row * K + k);
        }
        ok[g] = sl >= 0 && (int64_t)sl < p.n_slots;
        const uint4* xp = ex4 + (ok[g] ? (int64_t)sl * hv : 0);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int j = tid + v * blockDim.x;
          xv[g][v] = make_uint4(0u, 0u, 0u, 0u);
          if (ok[g] && j < sv) xv[g][v] = ld_stream(xp + j);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (ok[g]) {
#pragma unroll
          for (int v = 0; v < VPT; ++v) gate_add8(acc[v], gt[g], xv[g][v]);
        }
      }
    }
    if (row + gridDim.x >= p.T) pdl_trigger();

    uint4 ro[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * blockDim.x;
      if (j < sv) {
        const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        uint32_t red[4], out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          red[e] = pack_bf16x2(acc[k][2 * e], acc[k][2 * e + 1]);
          const float s0 = bf_lo(red[e]) + bf_lo(rw[e]);
          const float s1 = bf_hi(red[e]) + bf_hi(rw[e]);
          out[e] = pack_bf16x2(s0, s1);
          const float q0 = bf_lo(out[e]), q1 = bf_hi(out[e]);
          ss = fmaf(q0, q0, ss);
          ss = fmaf(q1, q1, ss);
        }
        st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j,
                  make_uint4(red[0], red[1], red[2], red[3]));
        ro[k] = make_uint4(out[0], out[1], out[2], out[3]);
        st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
      }
    }
    ss = warp_sum(ss);
    float* ws = warp_ss[it & 1];
    if (lane == 0) ws[warp] = ss;
    __syncthreads();
    float tot = sum_partials(ws, nwarps, lane);
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * blockDim.x;
      if (j < sv) {
        const uint4 wk = ld_keep(wv4 + j);
        const uint32_t q[4] = {ro[k].x, ro[k].y, ro[k].z, ro[k].w};
        const uint32_t w[4] = {wk.x, wk.y, wk.z, wk.w};
        uint32_t n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n0 = (bf_lo(q[e]) * rstd) * bf_lo(w[e]);
          const float n1 = (bf_hi(q[e]) * rstd) * bf_hi(w[e]);
          n[e] = pack_bf16x2(n0, n1);
        }
        st_stream(reinterpret_cast<uint4*>(p.norm_out) + base + j,
                  make_uint4(n[0], n[1], n[2], n[3]));
      }
    }
  }
}

// ------------------------------------------- bulk (TMA-staged) kernel
// Persistent and warp-specialised.  A row of hv 16-byte vectors is cut into
// nseg column segments of at most nct vectors (nct = the consumer threads).
// A stage of the shared-memory ring holds one segment of every input of a
// row: W+1 slots (x[0..W-1], then the residual) of p.stage_stride bytes.
// Warp 0 is the producer: it streams the segments of this CTA's rows, in
// order, into the ring -- per segment lane 0 waits for the stage to be free
// and posts one expect_tx on its "full" mbarrier, then lane r issues the
// cp.async.bulk copy (the TMA engine's bulk copy) of input r, so the W+1
// copies, completing on that barrier, go out side by side.  The other warps
// are the consumers: thread c owns
// vector c of every segment (vector k*nct + c of the row); per segment it
// waits once for the stage, adds the W staged vectors in rank order, reads
// the residual's, releases the stage (one arrival per warp on its "empty"
// mbarrier) and rounds and stores reduced and residual_out; after the row's
// last segment come the sum of squares and the normalisation, as in
// farn_vec_kernel.  A row costs each consumer warp nseg waits, whatever W
// is, and the ring keeps stages * (W+1) * stage_stride bytes in flight per
// CTA without holding registers.
//
// Every wait is bounded: after kWaitLimitNs of globaltimer time the
// waiting thread sets the CTA's abort flag and a bit in *p.err and
// returns; the other threads see the flag in their own waits and leave.
// The producer, once it has issued its last copy (or given up), always
// waits (bounded again) for the copies it may still have in flight before
// it exits, so no copy lands in the shared memory of a finished CTA.
constexpr uint32_t kBulkMaxStages = 16;
constexpr int kBulkMaxConsumers = 256;   // consumer threads per CTA
constexpr int kBulkThreads = 32 + kBulkMaxConsumers;
// The one- and two-segment builds take up to 512 consumer threads, used
// where the consumers set the pace: the MoE combine (three rounded
// operations per gathered element; GB300, K = 8, H = 7168, T = 4096: 98.7 %
// of the copy bandwidth with 448 consumer threads and 2 segments, 82.7 %
// with 320 and 3, 79.1 % with 224 and 4) and rank sums of W >= 8 inputs.
constexpr int kBulkMaxConsumersWide = 512;
constexpr int64_t kBulkMaxH = 16384;     // longest row the bulk plan takes
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr int kBulkErrFull = 1;     // consumer gave up waiting for a stage
constexpr int kBulkErrEmpty = 2;    // producer gave up waiting for a free stage
constexpr int kBulkErrReduce = 4;   // consumer gave up in the row reduction
constexpr int kBulkErrDrain = 8;    // producer gave up draining its copies

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completion counted in transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// Bounded phase wait.  false: gave up (time limit, or the CTA aborted).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag, int* err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(err, code);
      return false;
    }
  }
}

// Dynamic shared memory: [stages][W+1][stage_stride] ring, then the barriers.
struct BulkBarriers {
  uint64_t full[kBulkMaxStages];
  uint64_t empty[kBulkMaxStages];
  uint64_t reduce[2];          // per row parity: one arrival per consumer warp
  uint64_t never;              // nothing arrives on it (stall_test)
  float warp_ss[2][32];
  int abort_flag;
};

// VPT: the most segments per row (vectors per consumer thread) this
// instantiation takes.  The host guarantees H % 8 == 0, 16-byte aligned
// tensors, ceil(hv / nct) <= VPT, a stage_stride of at least nct * 16 bytes
// (a multiple of 128) and blockDim.x = 32 + nct with nct <= 256 (<= 512 at
// VPT <= 2).
// COMBINE: the MoE combine instead of the rank sum -- the W = K inputs of
// a row are the gathered expert rows expert_out[index[t,k]], summed as
// gates[t,k] * x with each product and sum rounded (slots outside
// [0, n_slots) are neither copied nor added); the producer warp's lane k
// and every consumer warp's lane k hold column k of the row's routing,
// loaded one of the CTA's rows ahead.
template <int VPT, bool COMBINE = false>
__global__ void __launch_bounds__(VPT <= 2 ? 32 + kBulkMaxConsumersWide : kBulkThreads, 1)
farn_bulk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t NS = p.stages;
  const uint32_t slot = p.stage_stride;
  const int W = p.W;
  const uint32_t stage_bytes = (uint32_t)(W + 1) * slot;
  BulkBarriers* bb = reinterpret_cast<BulkBarriers*>(smem + (size_t)NS * stage_bytes);
  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t full0 = (uint32_t)__cvta_generic_to_shared(&bb->full[0]);
  const uint32_t empty0 = (uint32_t)__cvta_generic_to_shared(&bb->empty[0]);
  const uint32_t reduce0 = (uint32_t)__cvta_generic_to_shared(&bb->reduce[0]);
  volatile int* abort_flag = &bb->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ncw = (int)(blockDim.x >> 5) - 1;          // consumer warps
  const int nct = ncw * 32;                            // consumer threads
  const int64_t hv = p.H >> 3;
  const int nseg = (int)((hv + nct - 1) / nct);        // segments per row
  const float Hf = (float)p.H;
  // MoE routing column `lane` of row r (-1 / 0 past the last row or column)
  auto load_slot = [&](int64_t r) -> int32_t {
    return (r < p.T && lane < W) ? __ldg(p.index + r * W + lane) : -1;
  };
  auto load_gate = [&](int64_t r) -> float {
    return (r < p.T && lane < W) ? __ldg(p.gates + r * W + lane) : 0.0f;
  };
  auto valid = [&](int32_t sl) { return sl >= 0 && (int64_t)sl < p.n_slots; };

  if (tid == 0) {
    for (uint32_t s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, (uint32_t)ncw);
    }
    mbar_init(reduce0, (uint32_t)ncw);
    mbar_init(reduce0 + 8, (uint32_t)ncw);
    mbar_init((uint32_t)__cvta_generic_to_shared(&bb->never), 1);
    bb->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // Lane 0 waits for a free stage and arms its "full" barrier; then lane
    // r issues the copy of input r (and r + 32), so the W+1 copies of a
    // segment are issued side by side rather than one after another.
    uint64_t q = 0;                       // segments issued so far
    bool ok = true;
    int32_t i_cur = -1, i_nxt = -1;       // MoE: this row's and the next row's slots
    if constexpr (COMBINE) {
      i_cur = load_slot(blockIdx.x);
      i_nxt = load_slot(blockIdx.x + gridDim.x);
    }
    for (int64_t row = blockIdx.x; row < p.T && ok; row += gridDim.x) {
      bool mine = false;                  // MoE: lane's slot is copied
      uint32_t ncopy = (uint32_t)(W + 1);
      if constexpr (COMBINE) {
        mine = lane < W && valid(i_cur);
        ncopy = (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, mine)) + 1;
      }
      for (int k = 0; k < nseg; ++k) {
        const uint32_t s = (uint32_t)(q % NS);
        const uint64_t n = q / NS;
        int good = 1;
        if (lane == 0 && n > 0)
          good = wait_phase(empty0 + 8 * s, (uint32_t)((n - 1) & 1), abort_flag, p.err,
                            kBulkErrEmpty) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, good, 0)) {
          ok = false;
          break;
        }
        const int64_t v0 = (int64_t)k * nct;
        const uint32_t bytes = (uint32_t)((hv - v0 < nct ? hv - v0 : nct) * 16);
        const int64_t off = (row * hv + v0) * 16;
        const uint32_t dst = ring + s * stage_bytes;
        if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * s, ncopy * bytes);
        __syncwarp();
        if constexpr (COMBINE) {
          if (mine)
            bulk_g2s(dst + (uint32_t)lane * slot,
                     reinterpret_cast<const unsigned char*>(p.expert_out) +
                         ((int64_t)i_cur * hv + v0) * 16,
                     bytes, full0 + 8 * s);
          if (lane == 0)
            bulk_g2s(dst + (uint32_t)W * slot,
                     reinterpret_cast<const unsigned char*>(p.residual) + off, bytes,
                     full0 + 8 * s);
        } else {
          for (int r = lane; r <= W; r += 32)
            bulk_g2s(dst + (uint32_t)r * slot,
                     reinterpret_cast<const unsigned char*>(r < W ? p.x[r] : p.residual) + off,
                     bytes, full0 + 8 * s);
        }
        ++q;
      }
      if constexpr (COMBINE) {
        i_cur = i_nxt;
        i_nxt = load_slot(row + 2 * (int64_t)gridDim.x);
      }
      if (row + gridDim.x >= p.T) pdl_trigger();
    }
    if (lane != 0) return;
    // Drain, always: the last min(q, NS) segments may still be in flight
    // (every earlier one was consumed before its stage was reused).
    const uint64_t first = q > NS ? q - NS : 0;
    for (uint64_t k = first; k < q; ++k) {
      const uint32_t s = (uint32_t)(k % NS);
      const uint32_t par = (uint32_t)((k / NS) & 1);
      if (mbar_try_wait(full0 + 8 * s, par)) continue;
      const uint64_t t0 = globaltimer_ns();
      bool done = false;
      while (!(done = mbar_try_wait(full0 + 8 * s, par)))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      if (!done) {
        atomicOr(p.err, kBulkErrDrain);
        break;
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  if (p.stall_test && blockIdx.x == 0) {
    // The test of the bounded waits: every consumer of CTA 0 waits on a
    // barrier nothing completes, the first past the time limit sets the
    // abort flag and kBulkErrFull, and all of them leave; the producer sees
    // the flag in its wait for a free stage, then drains its copies, which
    // all complete.  CTA 0's rows are left unwritten.
    wait_phase((uint32_t)__cvta_generic_to_shared(&bb->never), 0u, abort_flag, p.err,
               kBulkErrFull);
    return;
  }
  const int ctid = tid - 32;
  const int cw = warp - 1;
  // The weight slice stays in registers across rows (up to 8 segments);
  // longer rows read it again per row (it stays cached).
  constexpr bool kWeightRegs = VPT <= 8;
  uint4 wv[kWeightRegs ? VPT : 1];
  if constexpr (kWeightRegs) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t j = (int64_t)k * nct + ctid;
      if (k < nseg && j < hv) wv[k] = ld_keep(reinterpret_cast<const uint4*>(p.weight) + j);
    }
  }

  // MoE: this row's routing (c_*) and the CTA's next row's (n_*)
  int32_t c_sl = -1, n_sl = -1;
  float c_gt = 0.0f, n_gt = 0.0f;
  if constexpr (COMBINE) {
    c_sl = load_slot(blockIdx.x);
    c_gt = load_gate(blockIdx.x);
    n_sl = load_slot(blockIdx.x + gridDim.x);
    n_gt = load_gate(blockIdx.x + gridDim.x);
  }
  uint64_t q = 0;
  int it = 0;
  for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x, ++it) {
    const int64_t base = row * hv;
    uint4 ro[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (k < nseg) {
        const uint32_t s = (uint32_t)(q % NS);
        if (!wait_phase(full0 + 8 * s, (uint32_t)((q / NS) & 1), abort_flag, p.err,
                        kBulkErrFull))
          return;
        ++q;
        const int64_t j = (int64_t)k * nct + ctid;
        const bool in = j < hv;
        // this thread's vector in slot r of the stage
        const uint4* sv = reinterpret_cast<const uint4*>(smem + (size_t)s * stage_bytes) + ctid;
        const int sstep = (int)(slot >> 4);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = -0.0f;
        uint4 rv = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (COMBINE) {
          // gated sum of the gathered rows, k in order (the shuffles run on
          // every lane; only the reads and adds depend on `in`)
          for (int c = 0; c < W; ++c) {
            const int32_t sl = __shfl_sync(0xFFFFFFFFu, c_sl, c);
            const float g = __shfl_sync(0xFFFFFFFFu, c_gt, c);
            if (in && valid(sl)) gate_add8(acc, g, sv[c * sstep]);
          }
          if (in) rv = sv[W * sstep];
        } else if (in) {
          // a1: rank order, four staged vectors read ahead of their adds
          int r = 0;
          for (; r + 4 <= W; r += 4) {
            const uint4 v0 = sv[(r + 0) * sstep], v1 = sv[(r + 1) * sstep];
            const uint4 v2 = sv[(r + 2) * sstep], v3 = sv[(r + 3) * sstep];
            add8(acc, v0); add8(acc, v1); add8(acc, v2); add8(acc, v3);
          }
          for (; r < W; ++r) add8(acc, sv[r * sstep]);
          rv = sv[W * sstep];
        }
        // the stage's values are in registers: release it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (in) {
          // a2 + a5 and the thread's part of a3
          const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
          uint32_t red[4], out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            red[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
            const float s0 = bf_lo(red[e]) + bf_lo(rw[e]);
            const float s1 = bf_hi(red[e]) + bf_hi(rw[e]);
            out[e] = pack_bf16x2(s0, s1);
            const float q0 = bf_lo(out[e]), q1 = bf_hi(out[e]);
            ss = fmaf(q0, q0, ss);
            ss = fmaf(q1, q1, ss);
          }
          st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j,
                    make_uint4(red[0], red[1], red[2], red[3]));
          ro[k] = make_uint4(out[0], out[1], out[2], out[3]);
          st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
        }
      }
    }
    if (row + gridDim.x >= p.T) pdl_trigger();
    if constexpr (COMBINE) {
      c_sl = n_sl;
      c_gt = n_gt;
      n_sl = load_slot(row + 2 * (int64_t)gridDim.x);
      n_gt = load_gate(row + 2 * (int64_t)gridDim.x);
    }

    // a3: consumer-warp sums through shared memory, one mbarrier per row
    // parity (each consumer warp arrives once), combined by a butterfly.
    ss = warp_sum(ss);
    const int par = it & 1;
    if (lane == 0) {
      bb->warp_ss[par][cw] = ss;
      mbar_arrive(reduce0 + 8 * par);
    }
    if (!wait_phase(reduce0 + 8 * par, (uint32_t)((it >> 1) & 1), abort_flag, p.err,
                    kBulkErrReduce))
      return;
    const float tot = sum_partials(bb->warp_ss[par], ncw, lane);

    // a4
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t j = (int64_t)k * nct + ctid;
      if (k < nseg && j < hv) {
        uint4 wk;
        if constexpr (kWeightRegs) wk = wv[k];
        else wk = ld_keep(reinterpret_cast<const uint4*>(p.weight) + j);
        const uint32_t qv[4] = {ro[k].x, ro[k].y, ro[k].z, ro[k].w};
        const uint32_t w[4] = {wk.x, wk.y, wk.z, wk.w};
        uint32_t n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n0 = (bf_lo(qv[e]) * rstd) * bf_lo(w[e]);
          const float n1 = (bf_hi(qv[e]) * rstd) * bf_hi(w[e]);
          n[e] = pack_bf16x2(n0, n1);
        }
        st_stream(reinterpret_cast<uint4*>(p.norm_out) + base + j,
                  make_uint4(n[0], n[1], n[2], n[3]));
      }
    }
  }
}

// ------------------------------------------ stage (cp.async-staged) kernel
// Persistent; each thread stages its own 16-byte vectors.  The chunks of a
// CTA's rows, in order -- for each of its rows the row of x[0], ...,
// x[W-1], then of the residual -- flow through R private shared-memory
// slots per thread: the thread issues cp.async copies for chunk q+R while
// it adds chunk q, so R chunks of its vectors are in flight without
// holding registers, and the prefetch runs on across row boundaries while
// the CTA reduces a row.  A thread only ever reads the slots it filled
// itself, so the only waits are cp.async.wait_group (its own copies) and
// the row reduction's __syncthreads.  bf16 partials only: with fp32
// partials the register-staged farn_vec_kernel moves each row's twice
// larger partials at full bandwidth on its own.
//
// Shared memory: R * VPT * blockDim.x * 16 bytes, thread-interleaved so a
// warp's 16-byte accesses are contiguous.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// QM 1: also write the FP8 copy of norm_out (p.q_out, p.scale_out); QM 2:
// the NVFP4 copy (p.fp4_q, p.fp4_s); p.norm_out may then be null.  Each is
// compiled separately so the plain kernel is unchanged.
// The quantising kernels at 2 vectors per thread are built for two CTAs of
// 512 threads per SM (at most 64 registers per thread).
template <int VPT, int R, int QM = 0>
__global__ void __launch_bounds__(512, (VPT == 2 && QM != 0) ? 2 : 0)
farn_stage_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = (nt + 31) >> 5;
  const int64_t hv = p.H >> 3;
  const int W = p.W;
  const float Hf = (float)p.H;
  __shared__ float warp_ss[2][32];
  __shared__ float warp_mx[2][32];      // FP8 output only: row amax
  const uint32_t slots = (uint32_t)__cvta_generic_to_shared(smem);
  // slot s, vector k of this thread
  auto slot_addr = [&](int s, int k) -> uint32_t {
    return slots + (uint32_t)(((s * VPT + k) * nt + tid) * 16);
  };

  pdl_wait();
  // The weight slice stays in registers across rows, except in the FP8
  // build (64 registers for two CTAs of 512 threads per SM, where the
  // previous row's values are held for its pipelined amax): there it is
  // read again for every row from cache, which removes a register spill.
  constexpr bool kWeightRegs = QM != 1;
  uint4 wv[kWeightRegs ? VPT : 1];
  if constexpr (kWeightRegs) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) wv[k] = ld_keep(reinterpret_cast<const uint4*>(p.weight) + j);
    }
  }

  // Chunk cursor for issuing: (row, c); chunks run over this CTA's rows.
  int64_t irow = blockIdx.x;
  int ic = 0;
  auto issue_next = [&](int s) {
    if (irow < p.T) {
      const uint4* src = reinterpret_cast<const uint4*>(ic < W ? p.x[ic] : p.residual) +
                         irow * hv;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * nt;
        if (j < hv) cp_async16(slot_addr(s, k), src + j);
      }
      if (++ic > W) { ic = 0; irow += gridDim.x; }
    }
    cp_async_commit();   // one group per chunk, empty past the last row
  };
#pragma unroll
  for (int s = 0; s < R; ++s) issue_next(s);

  int q = 0;     // chunk being consumed
  int it = 0;
  int res_slot = 0;
  // FP8 output, pipelined: row i's amax is published at row i+1's
  // sum-of-squares barrier, so each row costs one barrier; the last row's
  // is published after the loop.
  uint4 nb_prev[VPT];
  float mx_prev = 0.0f;
  int64_t row_prev = -1;
  auto quant_store = [&](int64_t qrow, const float amax) {
    const float scale = e4m3_row_scale(amax);
    const float inv = e4m3_row_inv(amax);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) {
        const uint32_t n[4] = {nb_prev[k].x, nb_prev[k].y, nb_prev[k].z, nb_prev[k].w};
        uint32_t q8[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          q8[e] = pack_e4m3x2(bf_lo(n[e]) * inv, bf_hi(n[e]) * inv);
        asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};"
                     :: "l"(p.q_out + (qrow * hv + j) * 8), "r"(q8[0] | (q8[1] << 16)),
                        "r"(q8[2] | (q8[3] << 16)) : "memory");
      }
    }
    if (tid == 0) p.scale_out[qrow] = scale;
  };
  for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x, ++it) {
    const int64_t base = row * hv;
    float acc[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] = -0.0f;
    uint4 rv[VPT];
    // a1 in rank order, then the residual chunk.
    for (int c = 0; c <= W; ++c, ++q) {
      const int s = q % R;
      cp_async_wait<R - 1>();          // chunk q (the oldest group) has landed
      uint4 v[VPT];
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * nt;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (j < hv) v[k] = ld_shared_v4(slot_addr(s, k));
      }
      if (c < W) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          if constexpr (QM == 0) add8_x2(acc[k], v[k]);
          else add8(acc[k], v[k]);
        }
        // The adds consumed the slot's values: refill it.
        issue_next(s);
      } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) rv[k] = v[k];
        res_slot = s;
      }
    }
    if (row + gridDim.x >= p.T) pdl_trigger();

    uint4 ro[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) {
        const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        uint32_t red[4], out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          red[e] = pack_bf16x2(acc[k][2 * e], acc[k][2 * e + 1]);
          const float s0 = bf_lo(red[e]) + bf_lo(rw[e]);
          const float s1 = bf_hi(red[e]) + bf_hi(rw[e]);
          out[e] = pack_bf16x2(s0, s1);
          const float q0 = bf_lo(out[e]), q1 = bf_hi(out[e]);
          ss = fmaf(q0, q0, ss);
          ss = fmaf(q1, q1, ss);
        }
        st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j,
                  make_uint4(red[0], red[1], red[2], red[3]));
        ro[k] = make_uint4(out[0], out[1], out[2], out[3]);
        st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
      }
    }
    // The residual's slot is free once its values were used above.
    issue_next(res_slot);
    ss = warp_sum(ss);
    float* ws = warp_ss[it & 1];
    if (lane == 0) ws[warp] = ss;
    if constexpr (QM == 1) {
      if (row_prev >= 0) {
        const float m = warp_max(mx_prev);
        if (lane == 0) warp_mx[(it - 1) & 1][warp] = m;
      }
    }
    __syncthreads();
    // (The plain and NVFP4 kernels keep the serial sum over the warps: on
    // GB300 the butterfly measured no better there (prefill 102.7 % either
    // way, NVFP4 100.4 % against 100.7 %), while the FP8 kernel, which also
    // reduces the row's amax, went from 95.0 % to 97.1 % with it.)
    float tot = 0.0f;
    if constexpr (QM != 1) {
      for (int w = 0; w < nwarps; ++w) tot += ws[w];
    } else {
      tot = sum_partials(ws, nwarps, lane);
    }
    if constexpr (QM == 1) {
      if (row_prev >= 0) {
        const float* wm = warp_mx[(it - 1) & 1];
        float amax = max_partials(wm, nwarps, lane);
        quant_store(row_prev, amax);
      }
    }
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
    uint4 nb[VPT];
    float mx = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) {
        uint4 wk;
        if constexpr (kWeightRegs) wk = wv[k];
        else wk = ld_keep(reinterpret_cast<const uint4*>(p.weight) + j);
        const uint32_t qv[4] = {ro[k].x, ro[k].y, ro[k].z, ro[k].w};
        const uint32_t w[4] = {wk.x, wk.y, wk.z, wk.w};
        uint32_t n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n0 = (bf_lo(qv[e]) * rstd) * bf_lo(w[e]);
          const float n1 = (bf_hi(qv[e]) * rstd) * bf_hi(w[e]);
          n[e] = pack_bf16x2(n0, n1);
          if constexpr (QM == 1) mx = fmaxf(mx, fmaxf(fabsf(bf_lo(n[e])), fabsf(bf_hi(n[e]))));
        }
        if constexpr (QM != 0) nb[k] = make_uint4(n[0], n[1], n[2], n[3]);
        if (QM == 0 || p.norm_out)
          st_stream(reinterpret_cast<uint4*>(p.norm_out) + base + j,
                    make_uint4(n[0], n[1], n[2], n[3]));
      }
    }
    if constexpr (QM == 2) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * nt;
        uint32_t sb;
        const uint32_t codes = nvfp4_vec(j < hv ? nb[k] : make_uint4(0u, 0u, 0u, 0u), p.fp4_g, &sb);
        if (j < hv) {
          st_stream_u32(p.fp4_q + (base + j) * 4, codes);
          if ((j & 1) == 0) p.fp4_s[(base + j) >> 1] = (uint8_t)sb;
        }
      }
    }
    if constexpr (QM == 1) {
      // the row's amax (exact, NaN ignored) is reduced at the next row's
      // barrier, or after the loop for the last row
#pragma unroll
      for (int k = 0; k < VPT; ++k) nb_prev[k] = nb[k];
      mx_prev = mx;
      row_prev = row;
    }
  }
  if constexpr (QM == 1) {
    if (row_prev >= 0) {
      const float m = warp_max(mx_prev);
      if (lane == 0) warp_mx[(it - 1) & 1][warp] = m;
      __syncthreads();
      const float* wm = warp_mx[(it - 1) & 1];
      float amax = max_partials(wm, nwarps, lane);
      quant_store(row_prev, amax);
    }
  }
  cp_async_wait<0>();   // nothing may land after the CTA exits
}

// ------------------------------------ staged MoE combine (cp.async gather)
// The MoE combine for long inputs whose rows the TMA-staged kernel would
// split into more than two segments of fewer than 256 consumers, staged
// like farn_stage_kernel: each
// persistent CTA walks its rows; the chunks of a row are its K gathered
// expert rows (expert_out[index[t,k]]) and then its residual row; every
// thread keeps R chunks of its own 16-byte vectors in flight with
// cp.async.  A row's routing (K <= 32 slots and gates) lives in registers
// across the warp, lane k holding column k, and __shfl_sync hands column c
// to every lane; the issuing side and the consuming side each load it one
// of the CTA's rows ahead of use, so no chunk waits on an index load.  A
// slot outside [0, n_slots) issues no copy (only an empty group) and adds
// nothing; the consumer adds gate * x with the product and the sum each
// rounded (no fused multiply-add), k in order.  The two-vector build reads
// the weight again for every row (from cache) instead of holding it in
// registers: 56 registers, so two CTAs of 448 threads share an SM.
// Measured on GB300 (K = 8, H = 7168, T = 4096): 89.7 % of the copy
// bandwidth, against 88.3 % for the four-vector build holding the weight
// (126 registers, two CTAs of 224 threads), which itself falls to 80.9 %
// reading it per row; the two-vector build holding it needs 81 registers,
// one CTA per SM, 62.6 %.
template <int VPT, int R>
__global__ void __launch_bounds__(512)
farn_combine_stage_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = (nt + 31) >> 5;
  const int64_t hv = p.H >> 3;
  const int K = p.W;
  const int64_t step = gridDim.x;
  const float Hf = (float)p.H;
  __shared__ float warp_ss[2][32];
  const uint32_t slots = (uint32_t)__cvta_generic_to_shared(smem);
  const uint4* __restrict__ ex4 = reinterpret_cast<const uint4*>(p.expert_out);
  auto slot_addr = [&](int s, int k) -> uint32_t {
    return slots + (uint32_t)(((s * VPT + k) * nt + tid) * 16);
  };
  // Routing column `lane` of row r (-1 / 0 past the last row or column).
  auto load_slot = [&](int64_t r) -> int32_t {
    return (r < p.T && lane < K) ? __ldg(p.index + r * K + lane) : -1;
  };
  auto load_gate = [&](int64_t r) -> float {
    return (r < p.T && lane < K) ? __ldg(p.gates + r * K + lane) : 0.0f;
  };
  auto valid = [&](int32_t sl) { return sl >= 0 && (int64_t)sl < p.n_slots; };

  constexpr bool kWeightRegs = VPT >= 4;
  const uint4* __restrict__ wv4 = reinterpret_cast<const uint4*>(p.weight);
  pdl_wait();
  uint4 wv[kWeightRegs ? VPT : 1];
  if (kWeightRegs) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) wv[k] = ld_keep(wv4 + j);
    }
  }

  int64_t irow = blockIdx.x;
  int ic = 0;
  int32_t i_cur = load_slot(irow), i_nxt = load_slot(irow + step);
  // consumer's routing: this row (c_*) and the CTA's next row (n_*)
  int32_t c_sl = i_cur, n_sl = i_nxt;
  float c_gt = load_gate(irow), n_gt = load_gate(irow + step);
  auto issue_next = [&](int s) {
    if (irow < p.T) {                       // uniform across the CTA
      const uint4* src = nullptr;
      if (ic < K) {
        const int32_t sl = __shfl_sync(0xFFFFFFFFu, i_cur, ic);
        if (valid(sl)) src = ex4 + (int64_t)sl * hv;
      } else {
        src = reinterpret_cast<const uint4*>(p.residual) + irow * hv;
      }
      if (src) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int j = tid + k * nt;
          if (j < hv) cp_async16(slot_addr(s, k), src + j);
        }
      }
      if (++ic > K) {
        ic = 0;
        irow += step;
        i_cur = i_nxt;
        i_nxt = load_slot(irow + step);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < R; ++s) issue_next(s);

  int q = 0, it = 0, res_slot = 0;
  for (int64_t row = blockIdx.x; row < p.T; row += step, ++it) {
    const int64_t base = row * hv;
    float acc[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] = -0.0f;
    uint4 rv[VPT];
    for (int c = 0; c <= K; ++c, ++q) {
      const int s = q % R;
      cp_async_wait<R - 1>();
      if (c < K) {
        const int32_t sl = __shfl_sync(0xFFFFFFFFu, c_sl, c);
        const float gt = __shfl_sync(0xFFFFFFFFu, c_gt, c);
        if (valid(sl)) {
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            const int j = tid + k * nt;
            if (j < hv) gate_add8(acc[k], gt, ld_shared_v4(slot_addr(s, k)));
          }
        }
        issue_next(s);     // the adds above consumed the slot
      } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int j = tid + k * nt;
          rv[k] = make_uint4(0u, 0u, 0u, 0u);
          if (j < hv) rv[k] = ld_shared_v4(slot_addr(s, k));
        }
        res_slot = s;
      }
    }
    // the next row's routing is in registers; fetch the one after it
    c_sl = n_sl;
    c_gt = n_gt;
    n_sl = load_slot(row + 2 * step);
    n_gt = load_gate(row + 2 * step);
    if (row + step >= p.T) pdl_trigger();

    uint4 ro[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) {
        const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        uint32_t red[4], out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          red[e] = pack_bf16x2(acc[k][2 * e], acc[k][2 * e + 1]);
          const float s0 = bf_lo(red[e]) + bf_lo(rw[e]);
          const float s1 = bf_hi(red[e]) + bf_hi(rw[e]);
          out[e] = pack_bf16x2(s0, s1);
          const float q0 = bf_lo(out[e]), q1 = bf_hi(out[e]);
          ss = fmaf(q0, q0, ss);
          ss = fmaf(q1, q1, ss);
        }
        st_stream(reinterpret_cast<uint4*>(p.reduced) + base + j,
                  make_uint4(red[0], red[1], red[2], red[3]));
        ro[k] = make_uint4(out[0], out[1], out[2], out[3]);
        st_stream(reinterpret_cast<uint4*>(p.residual_out) + base + j, ro[k]);
      }
    }
    issue_next(res_slot);  // the residual's values were used above
    ss = warp_sum(ss);
    float* ws = warp_ss[it & 1];
    if (lane == 0) ws[warp] = ss;
    __syncthreads();
    float tot = 0.0f;                // serial over the warps (measured faster here)
    for (int w = 0; w < nwarps; ++w) tot += ws[w];
    const float rstd = 1.0f / sqrtf(tot / Hf + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * nt;
      if (j < hv) {
        const uint32_t qv[4] = {ro[k].x, ro[k].y, ro[k].z, ro[k].w};
        const uint4 wk = kWeightRegs ? wv[kWeightRegs ? k : 0] : ld_keep(wv4 + j);
        const uint32_t w[4] = {wk.x, wk.y, wk.z, wk.w};
        uint32_t n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n0 = (bf_lo(qv[e]) * rstd) * bf_lo(w[e]);
          const float n1 = (bf_hi(qv[e]) * rstd) * bf_hi(w[e]);
          n[e] = pack_bf16x2(n0, n1);
        }
        st_stream(reinterpret_cast<uint4*>(p.norm_out) + base + j,
                  make_uint4(n[0], n[1], n[2], n[3]));
      }
    }
  }
  cp_async_wait<0>();
}

}  // namespace farn
