// IVF-PQ list-scan kernel instantiations (split across files to keep
// compile units small).
#include "scan.cuh"

IVFPQ_INST_SCAN(0, 512)
IVFPQ_INST_SCAN(2, 512)
IVFPQ_INST_SCAN(4, 512)
IVFPQ_INST_SCAN(8, 512)
