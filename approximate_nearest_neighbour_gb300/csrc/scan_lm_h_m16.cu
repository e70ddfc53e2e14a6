// By-list list-scan kernels for m = 16 (see scan_lm.cuh): the filter pass
// with binary16 tables, 4 or 6 queries per item.
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(4, 8, 4, 0, IVFPQ_LUT_FP16)
IVFPQ_INST_SCAN_LM(4, 8, 6, 0, IVFPQ_LUT_FP16)
IVFPQ_INST_SCAN_LM(4, 4, 4, 0, IVFPQ_LUT_FP16)
IVFPQ_INST_SCAN_LM(4, 4, 6, 0, IVFPQ_LUT_FP16)
