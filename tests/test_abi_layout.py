"""The structures of the C ABI as a C compiler lays them out (include/amk.h,
compiled as C99 by gcc) against the Python binding's ctypes copies: every
field offset and every size.  A mismatch would make the binding pass
garbage across the boundary without any error."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pairs():
    import persistent_sm_decode_gb300 as amk
    return [(amk.Config, "amk_config"), (amk.LayerWeights, "amk_layer_weights"), (amk.Weights, "amk_weights"),
            (amk.ScheduleOptions, "amk_schedule_options"), (amk.PlanInfo, "amk_plan_info"),
            (amk.ErrorInfo, "amk_error_info")]


def test_binding_structures_match_the_c_header(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "amk.h"', '#include "amk_plan.h"',
             "int main(void) {"]
    for cls, cname in _pairs():
        lines.append('    printf("%s sizeof %%zu\\n", sizeof(%s));' % (cname, cname))
        for f, _ in cls._fields_:
            lines.append('    printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                           str(exe)])
    got = {}
    for ln in subprocess.check_output([str(exe)]).decode().splitlines():
        c, f, v = ln.split()
        got[(c, f)] = int(v)
    import ctypes
    for cls, cname in _pairs():
        assert got[(cname, "sizeof")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, "%s.%s" % (cname, f)


def test_headers_compile_as_plain_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "only.c"
    src.write_text('#include "amk.h"\n#include "amk_plan.h"\nint main(void) { return 0; }\n')
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I",
                           os.path.join(ROOT, "include"), str(src)])
