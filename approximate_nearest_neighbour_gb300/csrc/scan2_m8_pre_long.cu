// Register-codebook list-scan kernels for m = 8 with precomputed-term tables, warp queues of
// 128 / 256 entries (k > 256; see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(2, 12, 128, true)
IVFPQ_INST_SCAN2(2, 12, 256, true)
IVFPQ_INST_SCAN2(2, 8, 128, true)
IVFPQ_INST_SCAN2(2, 8, 256, true)
