/* nvtx_trace.c -- a minimal NVTX injection library for the tests.  The NVTX
 * loader in libzeroadam.so dlopens it from NVTX_INJECTION64_PATH at the
 * process's first NVTX call and calls InitializeInjectionNvtx2, which points
 * the range push/pop entries of NVTX's core function table at the recorders
 * below.  nvtx_trace_log() returns what was recorded: "+name;" for every range
 * pushed, "-;" for every range popped, in call order. */
#define NVTX_NO_IMPL
#include <nvtx3/nvToolsExt.h>
#include <string.h>

static char g_log[1 << 16];
static size_t g_len;

static void append(const char* s) {
  const size_t n = strlen(s);
  if (g_len + n + 1 >= sizeof(g_log)) return;
  memcpy(g_log + g_len, s, n);
  g_len += n;
  g_log[g_len] = 0;
}

static int NVTX_API record_push(const char* message) {
  append("+");
  append(message ? message : "(null)");
  append(";");
  return 0;
}

static int NVTX_API record_pop(void) {
  append("-;");
  return 0;
}

const char* nvtx_trace_log(void) { return g_log; }

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int last = 0; /* highest valid callback id of the module */
  if (cb == 0 || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &last)) return 0;
  if (table == 0 || last < NVTX_CBID_CORE_RangePop) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
