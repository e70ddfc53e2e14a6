// WarpSelect/BlockSelect kernel instantiations (split across files to
// keep compile units small).
#include "select_inst.cuh"

IVFPQ_INST_SELECT_PAIRS(2048, 4)
