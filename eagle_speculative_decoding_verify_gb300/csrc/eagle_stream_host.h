// Host-side workspace layout, cluster geometry and launch of the row stream
// (see eagle_rowstream.cuh), shared by the build and verify entry points.
#pragma once

#include "eagle_host.h"
#include "eagle_rowstream.cuh"

namespace eagle {

struct StreamLayout {
  int64_t n_rows;       // rows of all items
  int tiles_per_row;
  int rec_k;
  size_t off_item_cnt, off_rows, off_tiles, off_dec, total;
};

// header | item counters | row records | per-(row, tile, warp) sums |
// per-row decisions (verify)
inline StreamLayout stream_layout(int n_items, int rows_per_item, int vocab, int rec_k,
                                  bool tile_sums, bool decisions) {
  StreamLayout L;
  L.n_rows = static_cast<int64_t>(n_items) * rows_per_item;
  L.tiles_per_row = (vocab + kTile - 1) / kTile;
  L.rec_k = rec_k < 1 ? 1 : rec_k;
  size_t off = kWsHeader;
  L.off_item_cnt = off;
  off += sizeof(uint32_t) * static_cast<size_t>(n_items);
  off = align_up(off, 256);
  L.off_rows = off;
  off += static_cast<size_t>(rec_bytes(L.rec_k)) * static_cast<size_t>(L.n_rows);
  off = align_up(off, 256);
  L.off_tiles = off;
  if (tile_sums) off += sizeof(float2) * kWarps * static_cast<size_t>(L.n_rows) * L.tiles_per_row;
  off = align_up(off, 256);
  L.off_dec = off;
  if (decisions) off += sizeof(int2) * static_cast<size_t>(L.n_rows);
  L.total = align_up(off, 256);
  return L;
}

// Opt the kernel into the stream's shared memory; CTAs per SM (0 on error).
template <typename Args>
inline int stream_ctas_per_sm(void (*kernel)(Args)) {
  int occ = 0;
  const size_t smem = sizeof(StreamSmem);
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, smem) != cudaSuccess)
    return 0;
  return occ;
}

// attr: room for two attributes (cluster size; dependent launch)
inline cudaLaunchConfig_t stream_config(int64_t n_rows, int ctas, cudaStream_t stream,
                                        cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_rows * ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(StreamSmem);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attribute(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// CTAs per row (= cluster size): the largest size, at most kMaxCluster, at
// most one CTA per tile and at most the GPU's CTA slots per row, for which
// every row's cluster and `extra` more clusters are resident at once (one
// wave); 1 when no size gives one wave.  Returns 0 when the GPU cannot
// schedule the kernel at all.
template <typename Args>
inline int stream_ctas_per_row(void (*kernel)(Args), const StreamLayout& L, int ctas_per_sm,
                               int extra = 0) {
  const int64_t rows = (L.n_rows > 0 ? L.n_rows : 1) + extra;
  const int64_t slots = static_cast<int64_t>(sm_count()) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  int64_t p = slots / rows;
  if (p > kMaxCluster) p = kMaxCluster;
  if (p > L.tiles_per_row) p = L.tiles_per_row;
  if (p < 1) p = 1;
  bool any = false;
  for (int c = static_cast<int>(p); c >= 1; --c) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = stream_config(c, c, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    any |= n > 0;
    if (n >= rows) return c;
  }
  return any ? 1 : 0;
}

inline void fill_stream(RowStream& rs, const StreamLayout& L, char* ws, int n_items,
                        int rows_per_item, int vocab, int64_t row_stride, int ctas_per_row,
                        bool tile_sums) {
  rs.row_stride = row_stride;
  rs.n_items = n_items;
  rs.rows_per_item = rows_per_item;
  rs.vocab = vocab;
  rs.tiles_per_row = L.tiles_per_row;
  rs.ctas_per_row = ctas_per_row;
  rs.rec_k = L.rec_k;
  rs.err = reinterpret_cast<int32_t*>(ws);
  rs.item_cnt = reinterpret_cast<uint32_t*>(ws + L.off_item_cnt);
  rs.rows = ws + L.off_rows;
  rs.tile_sums = tile_sums ? reinterpret_cast<float2*>(ws + L.off_tiles) : nullptr;
}

template <typename Args>
inline eagle_status launch_stream(void (*kernel)(Args), const Args& A, int64_t n_rows, int ctas,
                                  cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = stream_config(n_rows, ctas, stream, attr);
  if (cudaLaunchKernelEx(&cfg, kernel, A) != cudaSuccess) {
    (void)cudaGetLastError();
    return EAGLE_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace eagle
