// Candidate selection kernels with long queues (k > 256), in their own
// translation units' worth of compile time.
#include "select_cand.cuh"

IVFPQ_INST_CAND(512)
IVFPQ_INST_CAND(1024)
IVFPQ_INST_CAND(2048)
