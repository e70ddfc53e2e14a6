// IVF-PQ list-scan kernel instantiations (split across files to keep
// compile units small).
#include "scan.cuh"

IVFPQ_INST_SCAN(0, 2048)
