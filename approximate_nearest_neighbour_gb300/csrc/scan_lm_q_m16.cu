// By-list list-scan kernels for m = 16 (see scan_lm.cuh): E4M3 tables, the
// filter pass with 4 or 8 queries per item and the bound pass (one query per
// item, per-lane queues of 2, 4 or 8 entries).
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(4, 8, 4, 0, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 8, 8, 0, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 4, 4, 0, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 4, 8, 0, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 8, 1, 2, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 8, 1, 4, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 8, 1, 8, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 4, 1, 2, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 4, 1, 4, IVFPQ_LUT_FP8)
IVFPQ_INST_SCAN_LM(4, 4, 1, 8, IVFPQ_LUT_FP8)
