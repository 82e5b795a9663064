// merge_cfg.cuh -- the two HBM-streaming kernels of the path.
//
// lse_merge: log-sum-exp merge of n partial attention results, the
//   recombination step of ring / Torus sequence-parallel attention
//   ("SwiftFusion: Scalable Sequence Parallelism ...", ideas 1-2):
//     M = max_c LSE_c,  LSE = M + ln sum_c exp(LSE_c - M),
//     out = sum_c exp(LSE_c - LSE) O_c,
//   partials with LSE_c = -inf are skipped (weight 0, never read).
// cfg_combine: out = eps_u + w (eps_c - eps_u), the join of the conditional
//   and unconditional paths of classifier-free guidance ("Accelerating
//   Diffusion via Hybrid Data-Pipeline Parallelism Based on Conditional
//   Guidance Scheduling", Technische Zusammenfassung 2A).
// cfg_combine_relmae: the same combine plus, in the same pass, the rel-MAE
//   discrepancy between the paths that the same page (2B) switches its
//   parallelism phases on: sum |eps_c - eps_u|, sum |eps_u| and their ratio.
//
// Both are pure streams: each output element is written once and each input
// element read once, 16 bytes per thread access, consecutive threads on
// consecutive addresses.  Grids are a multiple of the SM count with a
// grid-stride loop.  Each kernel lets the next one in the stream launch at
// once and waits for the previous one before its first memory access
// (programmatic dependent launch, see ptx.cuh).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace ditk {

constexpr int kStreamThreads = 256;

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }

// Row statistics: M = max, then LSE.  Returns -inf for an all -inf row.
__device__ __forceinline__ float merged_lse(const float *__restrict__ lses, int n, long long rows,
                                            long long r) {
  float mx = -INFINITY;
  for (int c = 0; c < n; ++c) mx = fmaxf(mx, __ldg(lses + c * rows + r));
  if (mx == -INFINITY) return -INFINITY;
  float z = 0.0f;
  for (int c = 0; c < n; ++c) {
    const float l = __ldg(lses + c * rows + r);
    if (l != -INFINITY) z += __expf(l - mx);
  }
  return mx + __logf(z);
}

// One thread per (row, 4 columns); D % 4 == 0 and 16-byte aligned pointers.
__global__ void __launch_bounds__(kStreamThreads)
    lse_merge_vec4_kernel(const float *__restrict__ partials, const float *__restrict__ lses, int n,
                          float *__restrict__ out, float *__restrict__ lse_out, long long rows, int d4) {
  griddep_launch_dependents();
  griddep_wait();
  const long long total = rows * d4;
  const long long stride = static_cast<long long>(gridDim.x) * kStreamThreads;
  for (long long idx = static_cast<long long>(blockIdx.x) * kStreamThreads + threadIdx.x; idx < total;
       idx += stride) {
    const long long r = idx / d4;
    const int c4 = static_cast<int>(idx - r * d4);
    const float lse = merged_lse(lses, n, rows, r);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != -INFINITY) {
      const float4 *src = reinterpret_cast<const float4 *>(partials) + r * d4 + c4;
      const long long cstride = rows * d4;
      // Loads issued for every chunk (the buffer is in bounds for all of
      // them) so that eight are in flight at once; an empty chunk's partial
      // is loaded but never used.
#pragma unroll 8
      for (int c = 0; c < n; ++c) {
        const float l = __ldg(lses + c * rows + r);
        const float4 v = ld_stream(src + c * cstride);
        if (l != -INFINITY) {
          const float w = __expf(l - lse);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
    st_stream(reinterpret_cast<float4 *>(out) + idx, acc);
    if (lse_out != nullptr && c4 == 0) lse_out[r] = lse;
  }
}

// As lse_merge_vec4_kernel, with the merged row rounded to bf16 (one 8-byte
// store per 4 columns): the second half of the chunk-parallel attention
// launch (dit_attn_fwd_split), writing the [B, H, S, D] bf16 output.
__global__ void __launch_bounds__(kStreamThreads)
    lse_merge_bf16_kernel(const float *__restrict__ partials, const float *__restrict__ lses, int n,
                          __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out, long long rows, int d4) {
  griddep_launch_dependents();
  griddep_wait();
  const long long total = rows * d4;
  const long long stride = static_cast<long long>(gridDim.x) * kStreamThreads;
  for (long long idx = static_cast<long long>(blockIdx.x) * kStreamThreads + threadIdx.x; idx < total;
       idx += stride) {
    const long long r = idx / d4;
    const int c4 = static_cast<int>(idx - r * d4);
    const float lse = merged_lse(lses, n, rows, r);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != -INFINITY) {
      const float4 *src = reinterpret_cast<const float4 *>(partials) + r * d4 + c4;
      const long long cstride = rows * d4;
#pragma unroll 8
      for (int c = 0; c < n; ++c) {
        const float l = __ldg(lses + c * rows + r);
        const float4 v = ld_stream(src + c * cstride);
        if (l != -INFINITY) {
          const float w = __expf(l - lse);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
    uint2 o;
    o.x = pack_bf16x2(acc.x, acc.y);
    o.y = pack_bf16x2(acc.z, acc.w);
    reinterpret_cast<uint2 *>(out)[idx] = o;
    if (lse_out != nullptr && c4 == 0) lse_out[r] = lse;
  }
}

// Fallback for D % 4 != 0: one thread per output element.
__global__ void __launch_bounds__(kStreamThreads)
    lse_merge_scalar_kernel(const float *__restrict__ partials, const float *__restrict__ lses, int n,
                            float *__restrict__ out, float *__restrict__ lse_out, long long rows, int D) {
  griddep_launch_dependents();
  griddep_wait();
  const long long total = rows * D;
  const long long stride = static_cast<long long>(gridDim.x) * kStreamThreads;
  for (long long idx = static_cast<long long>(blockIdx.x) * kStreamThreads + threadIdx.x; idx < total;
       idx += stride) {
    const long long r = idx / D;
    const int d = static_cast<int>(idx - r * D);
    const float lse = merged_lse(lses, n, rows, r);
    float acc = 0.0f;
    if (lse != -INFINITY) {
#pragma unroll 8
      for (int c = 0; c < n; ++c) {
        const float l = __ldg(lses + c * rows + r);
        const float v = __ldg(partials + (c * rows + r) * D + d);  // in bounds; unused if the chunk is empty
        if (l != -INFINITY) acc = fmaf(__expf(l - lse), v, acc);
      }
    }
    out[idx] = acc;
    if (lse_out != nullptr && d == 0) lse_out[r] = lse;
  }
}

// out may alias eps_c or eps_u: every element is read and then written by
// the same thread, so no __restrict__ here.
__global__ void __launch_bounds__(kStreamThreads)
    cfg_combine_vec4_kernel(const float4 *eps_c, const float4 *eps_u, float w, float4 *out, long long n4) {
  griddep_launch_dependents();
  griddep_wait();
  const long long stride = static_cast<long long>(gridDim.x) * kStreamThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kStreamThreads + threadIdx.x; i < n4; i += stride) {
    const float4 c = ld_stream(eps_c + i);
    const float4 u = ld_stream(eps_u + i);
    float4 o;
    o.x = fmaf(w, c.x - u.x, u.x);
    o.y = fmaf(w, c.y - u.y, u.y);
    o.z = fmaf(w, c.z - u.z, u.z);
    o.w = fmaf(w, c.w - u.w, u.w);
    st_stream(out + i, o);
  }
}

// rel-MAE = diff / base; an all-zero base gives 0 when diff is 0 too (the
// paths are identical) and +inf otherwise.  NaN inputs stay NaN.
__device__ __forceinline__ double relmae_ratio(double diff, double base) {
  return (base == 0.0 && diff == 0.0) ? 0.0 : diff / base;
}

// Sums of a (diff, base) pair over the block, added to sums[0..1] in fp64.
// sums[2] (zero on entry) counts the finished blocks while the grid runs; the
// last block to finish overwrites it with the ratio of the two totals.
__device__ __forceinline__ void block_add_sums(double diff, double base, double *sums) {
  __shared__ double red[2][kStreamThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    diff += __shfl_down_sync(0xffffffffu, diff, off);
    base += __shfl_down_sync(0xffffffffu, base, off);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = diff;
    red[1][warp] = base;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double d = 0.0, b = 0.0;
    for (int i = 0; i < kStreamThreads / 32; ++i) {
      d += red[0][i];
      b += red[1][i];
    }
    atomicAdd(sums, d);
    atomicAdd(sums + 1, b);
    __threadfence();
    unsigned long long *done = reinterpret_cast<unsigned long long *>(sums + 2);
    if (atomicAdd(done, 1ull) == gridDim.x - 1) {
      // Every other block's sums were added before its count.
      __threadfence();
      const double total_d = atomicAdd(sums, 0.0), total_b = atomicAdd(sums + 1, 0.0);
      sums[2] = relmae_ratio(total_d, total_b);
    }
  }
}

// One thread per float4 (grid-stride), the numel % 4 tail by the first
// threads; per-thread sums in fp32 (one accumulator per lane of the float4),
// fp64 from the warp level on.  sums[0..2] must be zero on entry.  out may alias
// eps_c or eps_u (each element is read and then written by the same thread).
__global__ void __launch_bounds__(kStreamThreads)
    cfg_combine_relmae_kernel(const float *eps_c, const float *eps_u, float w, float *out, long long numel,
                              double *sums) {
  griddep_launch_dependents();
  griddep_wait();
  const long long n4 = numel >> 2;
  const float4 *c4 = reinterpret_cast<const float4 *>(eps_c);
  const float4 *u4 = reinterpret_cast<const float4 *>(eps_u);
  float4 *o4 = reinterpret_cast<float4 *>(out);
  float4 dsum = make_float4(0.f, 0.f, 0.f, 0.f), bsum = make_float4(0.f, 0.f, 0.f, 0.f);
  const long long tid = static_cast<long long>(blockIdx.x) * kStreamThreads + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * kStreamThreads;
  auto step = [&](const float4 &c, const float4 &u, long long i) {
    const float dx = c.x - u.x, dy = c.y - u.y, dz = c.z - u.z, dw = c.w - u.w;
    st_stream(o4 + i, make_float4(fmaf(w, dx, u.x), fmaf(w, dy, u.y), fmaf(w, dz, u.z), fmaf(w, dw, u.w)));
    dsum.x += fabsf(dx);
    dsum.y += fabsf(dy);
    dsum.z += fabsf(dz);
    dsum.w += fabsf(dw);
    bsum.x += fabsf(u.x);
    bsum.y += fabsf(u.y);
    bsum.z += fabsf(u.z);
    bsum.w += fabsf(u.w);
  };
  // Two grid-stride elements per trip, both pairs of loads issued before
  // either is used: the running sums would otherwise keep one pair in flight.
  long long i = tid;
  for (; i + stride < n4; i += 2 * stride) {
    const float4 c0 = ld_stream(c4 + i), u0 = ld_stream(u4 + i);
    const float4 c1 = ld_stream(c4 + i + stride), u1 = ld_stream(u4 + i + stride);
    step(c0, u0, i);
    step(c1, u1, i + stride);
  }
  if (i < n4) step(ld_stream(c4 + i), ld_stream(u4 + i), i);
  double diff = (static_cast<double>(dsum.x) + dsum.y) + (static_cast<double>(dsum.z) + dsum.w);
  double base = (static_cast<double>(bsum.x) + bsum.y) + (static_cast<double>(bsum.z) + bsum.w);
  if (tid < numel - 4 * n4) {
    const long long i = 4 * n4 + tid;
    const float c = eps_c[i], u = eps_u[i];
    out[i] = fmaf(w, c - u, u);
    diff += fabsf(c - u);
    base += fabsf(u);
  }
  block_add_sums(diff, base, sums);
}

__global__ void cfg_combine_tail_kernel(const float *eps_c, const float *eps_u, float w, float *out,
                                        long long begin, long long numel) {
  griddep_launch_dependents();
  griddep_wait();
  const long long i = begin + threadIdx.x;
  if (i < numel) out[i] = fmaf(w, eps_c[i] - eps_u[i], eps_u[i]);
}

}  // namespace ditk
