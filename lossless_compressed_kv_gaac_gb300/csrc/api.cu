// Status names and the format version of the GAAC C ABI.
#include "gaac.h"

extern "C" const char* gaac_strerror(int status) {
  switch (status) {
    case GAAC_OK: return "ok";
    case GAAC_EINVAL: return "invalid argument";
    case GAAC_EPOOL: return "pool exhausted or index out of range";
    case GAAC_EFORMAT: return "malformed table entry or slot image";
    case GAAC_ECUDA: return "CUDA launch failed";
    case GAAC_ETIMEOUT: return "bounded wait in a kernel gave up";
    default: return "unknown status";
  }
}

extern "C" int gaac_format_version(void) { return 3; }
