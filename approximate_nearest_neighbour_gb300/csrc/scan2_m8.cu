// Register-codebook list-scan kernels for m = 8 (see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(2, 12, 32, false)
IVFPQ_INST_SCAN2(2, 12, 64, false)
IVFPQ_INST_SCAN2(2, 8, 32, false)
IVFPQ_INST_SCAN2(2, 8, 64, false)
