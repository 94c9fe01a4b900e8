// Parameters of the CUDA-core Q8_0 row kernels (matvec and small-M).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q8d {

// One Q8_0 matrix [p][n]; several matrices that read the same activations
// (q|k|v, gate|up) are processed by one launch.
struct RowSeg {
  const uint8_t* w;  // block stream, 16-byte aligned
  float* y;          // output row 0; row i of the output at y + i*ldy
  int p;             // output rows
  int reserved;
};

struct RowsParams {
  RowSeg seg[3];
  int nseg;
  int n;               // input dim (multiple of 32)
  const float* X;      // activations, row i at X + i*ldx, 16-byte aligned
  int ldx;
  int ldy;
  int m;               // activation rows (1 = matvec)
  int* d_err;          // device error word or nullptr
  // filled by the planner
  int bpr;
  long long row_bytes;
  long long vbegin[3];     // first virtual row of each matrix (concatenated rows)
  long long total_rows;    // sum of p
  long long rows_per_cta;  // contiguous virtual rows owned by one CTA
  int rows_per_tile, stage_bytes, nstages, segs_per_row;
  // matvec kernel (q8d_gemv.cu) only
  int paired;              // 1: warp pairs own the even / odd block columns of 64-column segments
  int win;                 // tiles per reduction window
  int win_rows;            // rows per window buffer (win * rows_per_tile)
  int np;                  // row pairs per warp per tile
};

// Plans tiles/stages and launches the kernel on `stream`.  Returns a status;
// *grid_out (if given) receives the number of CTAs launched.
int rows_plan_and_launch(RowsParams P, cudaStream_t stream, int* grid_out = nullptr);

// The m == 1 kernel (q8d_gemv.cu); P has bpr, row_bytes, vbegin and
// total_rows filled.  Q8D_EUNSUPPORTED when the rows are too long for it.
int gemv_plan_and_launch(RowsParams P, cudaStream_t stream, int* grid_out);

// The m == 1 tensor-core kernel (q8d_gemv_mma.cu) for one matrix with
// n % 256 == 0 and enough rows; Q8D_EUNSUPPORTED otherwise.
int gemv_mma_plan_and_launch(const RowsParams& P, cudaStream_t stream, int* grid_out);

}  // namespace q8d
