// WarpSelect/BlockSelect kernel instantiations (split across files to
// keep compile units small).
#include "select_inst.cuh"

IVFPQ_INST_SELECT_ROWS(512, 4)
