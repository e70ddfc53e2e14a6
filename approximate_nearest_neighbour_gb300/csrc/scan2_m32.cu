// Register-codebook list-scan kernels for m = 32 (see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(8, 3, 32, false)
IVFPQ_INST_SCAN2(8, 3, 64, false)
IVFPQ_INST_SCAN2(8, 4, 32, false)
IVFPQ_INST_SCAN2(8, 4, 64, false)
