// Device-side gather of the scheduled target rows out of page-locked host
// memory (internal header).
#pragma once

#include "common.cuh"

namespace spec {

struct GatherRowsParams {
  int R, G1;                 // requests; rows per request in the padded source (gamma + 1)
  size_t row_bytes;          // V * element size
  const unsigned char* src;  // device address of the host array [R, G1] rows
  unsigned char* dst;        // packed rows [row_off[R]] of the verify batch
  const int32_t* row_off;    // [R + 1] packed row offsets from the schedule
  uint32_t* status;
};

// Rows 1 .. row_off[r + 1] - row_off[r] of every request r, copied from
// src[r][j - 1] to dst[row_off[r] + j - 1].
cudaError_t launch_gather_rows(const GatherRowsParams& p, cudaStream_t stream);

}  // namespace spec
