/* A minimal NVTX v3 injection library for the tracing test: it takes over
 * the core RangePushA / RangePop callbacks and appends one line per event to
 * the file named by OSCAR_NVTX_LOG ("push <name>" or "pop").  Loaded by the
 * NVTX implementation inside liboscar.so when NVTX_INJECTION64_PATH names
 * it; it uses only the documented export-table handshake of the NVTX v3
 * headers. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log = NULL;

static int record_push(const char* message) {
  if (g_log) {
    fprintf(g_log, "push %s\n", message ? message : "");
    fflush(g_log);
  }
  return 0;
}

static int record_pop(void) {
  if (g_log) {
    fputs("pop\n", g_log);
    fflush(g_log);
  }
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
  const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = NULL;
  unsigned int size = 0;
  const char* path = getenv("OSCAR_NVTX_LOG");
  if (!cb || !path || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
  if (size <= NVTX_CBID_CORE_RangePop) return 0;
  g_log = fopen(path, "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
