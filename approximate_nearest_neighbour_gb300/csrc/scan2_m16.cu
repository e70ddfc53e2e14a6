// Register-codebook list-scan kernels for m = 16 (see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(4, 8, 32, false)
IVFPQ_INST_SCAN2(4, 8, 64, false)
IVFPQ_INST_SCAN2(4, 4, 32, false)
IVFPQ_INST_SCAN2(4, 4, 64, false)
