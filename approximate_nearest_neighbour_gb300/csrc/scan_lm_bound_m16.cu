// List-major bound pass for m = 16 (see scan_lm.cuh): one query per item,
// per-lane queues of 2, 4 or 8 entries.
#include "scan_lm.cuh"

IVFPQ_INST_SCAN_LM(4, 8, 1, 2)
IVFPQ_INST_SCAN_LM(4, 8, 1, 4)
IVFPQ_INST_SCAN_LM(4, 8, 1, 8)
IVFPQ_INST_SCAN_LM(4, 4, 1, 2)
IVFPQ_INST_SCAN_LM(4, 4, 1, 4)
IVFPQ_INST_SCAN_LM(4, 4, 1, 8)
