// Register-codebook list-scan kernels for m = 8 with precomputed-term tables (see scan2.cuh).
#include "scan2.cuh"

IVFPQ_INST_SCAN2(2, 12, 32, true)
IVFPQ_INST_SCAN2(2, 12, 64, true)
IVFPQ_INST_SCAN2(2, 8, 32, true)
IVFPQ_INST_SCAN2(2, 8, 64, true)
