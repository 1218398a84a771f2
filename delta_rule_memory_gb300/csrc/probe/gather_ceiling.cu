// gather_ceiling.cu - measurement probe, not part of libsdm: the DRAM
// throughput of random row-piece gathers and scatters on a table laid out as
// the sparse memory's (rows of 3840 bytes = 960 fp32, 3.54 GB in all), as a
// function of the piece size.  This is the access pattern of the sparse scan
// (every token reads W + R rows and writes W rows of a column tile), without
// its arithmetic or its per-token dependency chain.
//
// Each warp step reads UNROLL x (32 / G) pieces of G float4 (16 G bytes,
// G consecutive lanes per piece) from rows drawn by a hash, so no index array
// is read, and in the 2 : 1 mode writes one piece for every two read.  With
// ADJ the 4 warps of a CTA take the 4 adjacent pieces of the same rows at the
// same step, like the scan's 4 column-tile warps of one CTA.
//
// Build and run:  nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o probe gather_ceiling.cu && ./probe
// (bench.py --probe gather does both).  Prints one JSON object per case.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

namespace {

constexpr int kRowF4 = 240;  // float4 per row
constexpr int kUnroll = 8;

__device__ __forceinline__ uint32_t mix(uint32_t x) {  // an integer hash (xor-shift-multiply)
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int G, bool WRITE, bool ADJ>
__global__ void __launch_bounds__(256) probe_kernel(float4 *__restrict__ tab, uint32_t nrows, int iters,
                                                    float4 *__restrict__ sink) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t gw = blockIdx.x * 8 + warp;
  const int grp = lane / G, q = lane % G;
  constexpr int kTiles = kRowF4 / G;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int it = 0; it < iters; ++it) {
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // ADJ: one row per (CTA, warp pair group), the warp picks piece warp % 4 of an aligned run of 4
      const uint32_t key = ADJ ? ((blockIdx.x * 2 + warp / 4) * iters + it) * kUnroll * 32 + u * 32 + grp
                               : (gw * iters + it) * kUnroll * 32 + u * 32 + grp;
      const uint32_t h = mix(key);
      const uint32_t row = h % nrows;
      const uint32_t tile = ADJ ? 4 * ((h >> 20) % (kTiles / 4)) + (warp & 3) : (h >> 20) % kTiles;
      v[u] = __ldcg(tab + static_cast<size_t>(row) * kRowF4 + tile * G + q);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      acc.x += v[u].x;
      acc.y += v[u].y;
      acc.z += v[u].z;
      acc.w += v[u].w;
    }
    if (WRITE) {
#pragma unroll
      for (int u = 0; u < kUnroll / 2; ++u) {
        const uint32_t key = ADJ ? ~(((blockIdx.x * 2 + warp / 4) * iters + it) * kUnroll * 32 + u * 32 + grp)
                                 : ~((gw * iters + it) * kUnroll * 32 + u * 32 + grp);
        const uint32_t h = mix(key);
        const uint32_t row = h % nrows;
        const uint32_t tile = ADJ ? 4 * ((h >> 20) % (kTiles / 4)) + (warp & 3) : (h >> 20) % kTiles;
        tab[static_cast<size_t>(row) * kRowF4 + tile * G + q] = v[u];
      }
    }
  }
  if (acc.x == 1234.5f) sink[0] = acc;  // keeps the loads
}

template <int G, bool WRITE, bool ADJ>
int run(float4 *tab, uint32_t nrows, float4 *sink, int blocks, int iters) {
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  for (int w = 0; w < 3; ++w) probe_kernel<G, WRITE, ADJ><<<blocks, 256>>>(tab, nrows, iters, sink);
  const int reps = 10;
  cudaEventRecord(a);
  for (int r = 0; r < reps; ++r) probe_kernel<G, WRITE, ADJ><<<blocks, 256>>>(tab, nrows, iters, sink);
  cudaEventRecord(b);
  if (cudaEventSynchronize(b) != cudaSuccess) return 1;
  float ms = 0.f;
  cudaEventElapsedTime(&ms, a, b);
  ms /= reps;
  const double pieces = static_cast<double>(blocks) * 8 * iters * kUnroll * (32 / G);
  const double bytes = pieces * 16 * G * (WRITE ? 1.5 : 1.0);
  printf("{\"probe\": \"random row-piece gather%s\", \"piece_bytes\": %d, \"adjacent_4_warps\": %s, "
         "\"ctas\": %d, \"ms\": %.3f, \"GB_per_s\": %.0f}\n",
         WRITE ? " + scatter (2 reads : 1 write)" : " (reads only)", 16 * G, ADJ ? "true" : "false", blocks, ms,
         bytes / ms / 1e6);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return 0;
}

}  // namespace

int main() {
  const uint32_t nrows = 16u * 57600u;  // B*H = 16 tables of N = 57,600 rows: 3.54 GB
  float4 *tab = nullptr, *sink = nullptr;
  if (cudaMalloc(&tab, static_cast<size_t>(nrows) * kRowF4 * sizeof(float4)) != cudaSuccess ||
      cudaMalloc(&sink, sizeof(float4)) != cudaSuccess) {
    printf("{\"error\": \"allocation failed\"}\n");
    return 1;
  }
  cudaMemset(tab, 0, static_cast<size_t>(nrows) * kRowF4 * sizeof(float4));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = sms * 8, iters = 512;
  int rc = 0;
  rc |= run<4, false, false>(tab, nrows, sink, blocks, iters);
  rc |= run<4, true, false>(tab, nrows, sink, blocks, iters);
  rc |= run<4, true, true>(tab, nrows, sink, blocks, iters);
  rc |= run<8, true, false>(tab, nrows, sink, blocks, iters);
  rc |= run<16, true, false>(tab, nrows, sink, blocks, iters);
  rc |= run<16, false, false>(tab, nrows, sink, blocks, iters);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess || rc) {
    printf("{\"error\": \"%s\"}\n", cudaGetErrorString(e));
    return 1;
  }
  cudaFree(tab);
  cudaFree(sink);
  return 0;
}
