// By-list list-scan kernels for m = 16 (see scan_lm.cuh): the filter pass
// with fp32 tables, 2 or 3 queries per item.
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(4, 8, 2, 0, IVFPQ_LUT_FP32)
IVFPQ_INST_SCAN_LM(4, 8, 3, 0, IVFPQ_LUT_FP32)
IVFPQ_INST_SCAN_LM(4, 4, 2, 0, IVFPQ_LUT_FP32)
IVFPQ_INST_SCAN_LM(4, 4, 3, 0, IVFPQ_LUT_FP32)
