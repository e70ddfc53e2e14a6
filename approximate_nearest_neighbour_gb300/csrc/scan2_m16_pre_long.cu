// Register-codebook list-scan kernels for m = 16 with precomputed-term tables, warp queues of
// 128 / 256 entries (k > 256; see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(4, 8, 128, true)
IVFPQ_INST_SCAN2(4, 8, 256, true)
IVFPQ_INST_SCAN2(4, 4, 128, true)
IVFPQ_INST_SCAN2(4, 4, 256, true)
