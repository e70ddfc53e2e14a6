// List-major list-scan kernels for m = 8 (see scan_lm.cuh): the filter pass
// with 2 or 3 queries per table set.
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(2, 12, 2, 0)
IVFPQ_INST_SCAN_LM(2, 12, 3, 0)
IVFPQ_INST_SCAN_LM(2, 8, 2, 0)
IVFPQ_INST_SCAN_LM(2, 8, 3, 0)
