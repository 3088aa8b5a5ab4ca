// Online-softmax merge of normalised partial attention outputs.
//
// Every rank folds the partial results of the blocks it meets into one
// answer with the online-softmax rule ("day 83" blog, "Context parallelism:
// splitting the sequence"); this kernel is that fold over n partials.  For
// n partials (O_i, LSE_i) of the same query row:
//   M = max_i LSE_i,  w_i = exp(LSE_i - M),  LSE = M + ln sum_i w_i,
//   O = sum_i w_i O_i / sum_i w_i;   all LSE_i = -inf  ->  O = 0, LSE = -inf.
//
// HBM-bound: every partial byte is read once.  A row of d fp32 values is
// d/4 lanes x 16 bytes, so a warp reads whole 512-byte (d = 128) or two
// 256-byte (d = 64) rows per partial with 128-bit streaming loads.  For
// n <= 8 every lane holds the row's LSEs and eight 16-byte partial loads in
// registers before any arithmetic (all loads in flight together) and the grid
// strides over rows; larger n takes a loop of eight partials at a time.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float4 ld_stream(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Fast path for n <= 8 partials: every lane keeps the row's LSEs in
// registers and a warp merges ROWS rows per iteration, so 8 * ROWS 16-byte
// loads per lane are in flight; grid-stride over rows.
template <int D, int ROWS>
__global__ void __launch_bounds__(256) lse_merge_kernel8(const float *__restrict__ o_parts,
                                                         const float *__restrict__ lse_parts,
                                                         int n, int64_t rows,
                                                         __nv_bfloat16 *__restrict__ out,
                                                         float *__restrict__ lse_out,
                                                         int *status) {
  constexpr int kLanes = D / 4;  // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanes;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t part_stride = rows * kLanes;  // float4 per partial
  for (int64_t base = warp0 * kRowsPerWarp * ROWS; base < rows;
       base += warps * kRowsPerWarp * ROWS) {
    float4 v[ROWS][8];
    float l[ROWS][8];
    int64_t row[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      row[r] = base + r * kRowsPerWarp + lane / kLanes;
      const bool ok = row[r] < rows && RA_IN_BOUNDS(n <= 8 && sub < kLanes, status);
      const float4 *src = reinterpret_cast<const float4 *>(o_parts) + row[r] * kLanes + sub;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (ok && u < n) {
          l[r][u] = __ldg(lse_parts + static_cast<int64_t>(u) * rows + row[r]);
          v[r][u] = ld_stream(src + static_cast<int64_t>(u) * part_stride);
        } else {
          l[r][u] = -INFINITY;
          v[r][u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      if (row[r] >= rows) continue;
      float M = l[r][0];
#pragma unroll
      for (int u = 1; u < 8; ++u) M = fmaxf(M, l[r][u]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float wt = fast_ex2((l[r][u] - M) * kLog2e);  // -inf -> 0
          W += wt;
          acc.x = fmaf(wt, v[r][u].x, acc.x);
          acc.y = fmaf(wt, v[r][u].y, acc.y);
          acc.z = fmaf(wt, v[r][u].z, acc.z);
          acc.w = fmaf(wt, v[r][u].w, acc.w);
        }
      }
      const float inv = (W > 0.f) ? 1.f / W : 0.f;
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t *>(&lo);
      packed.y = *reinterpret_cast<uint32_t *>(&hi);
      reinterpret_cast<uint2 *>(out)[row[r] * kLanes + sub] = packed;
      if (sub == 0) lse_out[row[r]] = (W > 0.f) ? M + fast_lg2(W) * kLn2 : -INFINITY;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float *__restrict__ o_parts,
                                                        const float *__restrict__ lse_parts,
                                                        int n, int64_t rows,
                                                        __nv_bfloat16 *__restrict__ out,
                                                        float *__restrict__ lse_out,
                                                        int *status) {
  constexpr int kLanes = D / 4;            // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanes;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t row = warp_global * kRowsPerWarp + lane / kLanes;
  if (row >= rows || !RA_IN_BOUNDS(row >= 0 && sub < kLanes, status)) return;

  float M = -INFINITY;
  for (int i = 0; i < n; ++i) M = fmaxf(M, __ldg(lse_parts + static_cast<int64_t>(i) * rows + row));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    const float4 *src = reinterpret_cast<const float4 *>(o_parts) + row * kLanes + sub;
    const int64_t part_stride = rows * kLanes;  // float4 per partial
    for (int i0 = 0; i0 < n; i0 += 8) {
      float4 v[8];
      float wt[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u < n) {
          v[u] = ld_stream(src + static_cast<int64_t>(i0 + u) * part_stride);
          wt[u] = fast_ex2((__ldg(lse_parts + static_cast<int64_t>(i0 + u) * rows + row) - M) *
                           kLog2e);
        } else {
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          wt[u] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        W += wt[u];
        acc.x = fmaf(wt[u], v[u].x, acc.x);
        acc.y = fmaf(wt[u], v[u].y, acc.y);
        acc.z = fmaf(wt[u], v[u].z, acc.z);
        acc.w = fmaf(wt[u], v[u].w, acc.w);
      }
    }
  }
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t *>(&lo);
  packed.y = *reinterpret_cast<uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(out)[row * kLanes + sub] = packed;
  if (sub == 0) lse_out[row] = (W > 0.f) ? M + fast_lg2(W) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int n, int64_t rows,
                             int d, void *out, float *lse_out, int *status,
                             cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (status == nullptr) return cudaErrorInvalidValue;
  if (n <= 8) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    constexpr int kRows = 1;
    const int64_t rows_per_block = (256 / 32) * (d == 128 ? 1 : 2) * kRows;
    const int64_t want = (rows + rows_per_block - 1) / rows_per_block;
    const int grid = static_cast<int>(want < sms * 8 ? want : sms * 8);
    if (d == 128)
      lse_merge_kernel8<128, kRows><<<grid, 256, 0, stream>>>(
          o_parts, lse_parts, n, rows, static_cast<__nv_bfloat16 *>(out), lse_out, status);
    else
      lse_merge_kernel8<64, kRows><<<grid, 256, 0, stream>>>(
          o_parts, lse_parts, n, rows, static_cast<__nv_bfloat16 *>(out), lse_out, status);
    return cudaGetLastError();
  }
  const int rows_per_block = (256 / 32) * (d == 128 ? 1 : 2);
  const int64_t grid = (rows + rows_per_block - 1) / rows_per_block;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  if (d == 128)
    lse_merge_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
        o_parts, lse_parts, n, rows, static_cast<__nv_bfloat16 *>(out), lse_out, status);
  else
    lse_merge_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
        o_parts, lse_parts, n, rows, static_cast<__nv_bfloat16 *>(out), lse_out, status);
  return cudaGetLastError();
}

}  // namespace ra
