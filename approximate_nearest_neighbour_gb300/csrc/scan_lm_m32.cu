// List-major list-scan kernels for m = 32 (see scan_lm.cuh): the filter pass
// with 2 or 3 queries per table set.
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(8, 3, 2, 0)
IVFPQ_INST_SCAN_LM(8, 3, 3, 0)
IVFPQ_INST_SCAN_LM(8, 4, 2, 0)
IVFPQ_INST_SCAN_LM(8, 4, 3, 0)
