// Host-side geometry and workspace layout of the row stream (see
// eagle_rowstream.cuh), shared by the build and verify entry points.
#pragma once

#include "eagle_host.h"
#include "eagle_rowstream.cuh"

namespace eagle {

struct StreamLayout {
  int64_t n_rows;       // rows of all items
  int tiles_per_row;
  int64_t total_tiles;
  int rec_k;
  size_t off_row_cnt, off_item_cnt, off_pieces, off_rows, off_tiles, total;
};

inline StreamLayout stream_layout(int n_items, int rows_per_item, int vocab, int rec_k,
                                  bool tile_sums) {
  StreamLayout L;
  L.n_rows = static_cast<int64_t>(n_items) * rows_per_item;
  L.tiles_per_row = (vocab + kTile - 1) / kTile;
  L.total_tiles = L.n_rows * L.tiles_per_row;
  L.rec_k = rec_k < 1 ? 1 : rec_k;
  const size_t rb = static_cast<size_t>(rec_bytes(L.rec_k));
  size_t off = kWsHeader;
  L.off_row_cnt = off;
  off += sizeof(uint32_t) * static_cast<size_t>(L.n_rows);
  L.off_item_cnt = off;
  off += sizeof(uint32_t) * static_cast<size_t>(n_items);
  off = align_up(off, 256);
  L.off_pieces = off;
  off += rb * kMaxPieces * static_cast<size_t>(L.n_rows);
  off = align_up(off, 256);
  L.off_rows = off;
  off += rb * static_cast<size_t>(L.n_rows);
  off = align_up(off, 256);
  L.off_tiles = off;
  if (tile_sums) off += sizeof(float2) * kWarps * static_cast<size_t>(L.total_tiles);
  L.total = align_up(off, 256);
  return L;
}

// Grid: whole CTAs per SM, no more CTAs than tiles, and few enough CTAs per
// row that a row has at most kMaxPieces pieces.
inline int stream_grid(const StreamLayout& L, int ctas_per_sm) {
  int64_t G = static_cast<int64_t>(sm_count()) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  if (G < 1) G = 1;
  if (G > L.total_tiles) G = L.total_tiles;
  const int64_t TR = L.tiles_per_row;
  for (;;) {
    const int64_t per = L.total_tiles / G;  // every CTA owns >= per tiles
    const int64_t pieces = (TR + per - 1) / per + 1;
    if (pieces <= kMaxPieces || G == 1) break;
    --G;
  }
  return static_cast<int>(G);
}

inline void fill_stream(RowStream& rs, const StreamLayout& L, char* ws, int n_items,
                        int rows_per_item, int vocab, int64_t row_stride, int grid,
                        bool tile_sums) {
  rs.row_stride = row_stride;
  rs.total_tiles = L.total_tiles;
  rs.n_items = n_items;
  rs.rows_per_item = rows_per_item;
  rs.vocab = vocab;
  rs.tiles_per_row = L.tiles_per_row;
  rs.grid = grid;
  rs.max_pieces = kMaxPieces;
  rs.rec_k = L.rec_k;
  rs.err = reinterpret_cast<int32_t*>(ws);
  rs.row_cnt = reinterpret_cast<uint32_t*>(ws + L.off_row_cnt);
  rs.item_cnt = reinterpret_cast<uint32_t*>(ws + L.off_item_cnt);
  rs.pieces = ws + L.off_pieces;
  rs.rows = ws + L.off_rows;
  rs.tile_sums = tile_sums ? reinterpret_cast<float2*>(ws + L.off_tiles) : nullptr;
}

}  // namespace eagle
