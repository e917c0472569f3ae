// Host-side launch helpers shared by the kernel files: the segment table a kernel receives by value, and
// grid sizes of whole waves of resident CTAs.
#pragma once

#include <cuda_runtime.h>

#include "dp_device.cuh"
#include "dp_internal.h"

namespace dp {

// Streaming multiprocessors of the current device (cached per device; 148 if the query fails).
inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

// The plan's segments as the kernels' by-value table (e[nseg] is the sentinel).
template <int MAXSEG>
void fill_seg(SegTable<MAXSEG>& T, const Plan& P) {
  T.psi = P.psi;
  T.nseg = P.nseg;
  T.ntiles = P.ntiles;
  for (int k = 0; k <= P.nseg; ++k) {
    T.e[k].goff = P.e[k].goff;
    T.e[k].loff = P.e[k].loff;
    T.e[k].tile0 = P.e[k].tile0;
    T.e[k].owner = P.e[k].owner;
  }
}

// One wave of resident CTAs (SMs x CTAs per SM), capped by the tile count; at least 1, since every CTA of a
// reduction joins its grid-wide finish.
template <typename K>
int occupancy_grid(K kernel, int threads, size_t smem, int ntiles) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  long long g = (long long)sm_count() * per_sm;
  if (ntiles < g) g = ntiles;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace dp
