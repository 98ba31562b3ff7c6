"""Host checks of the build's ptxas gates: the forward kernel's register count (its setmaxnreg
split assumes the launch holds exactly FWD_LAUNCH_REGISTERS per thread) and the kernels that
must compile without register spills."""
import pytest

from exact_attention_49_gb300 import build

REPORT = """
ptxas info    : Compiling entry function '_ZN2fa10fwd_kernelILi128ELi0ELb0EEEv14CUtensorMap_stS1_S1_NS_9FwdParamsEi' for 'sm_103a'
ptxas info    : Function properties for _ZN2fa10fwd_kernelILi128ELi0ELb0EEEv14CUtensorMap_stS1_S1_NS_9FwdParamsEi
    %s bytes stack frame, %s bytes spill stores, %s bytes spill loads
ptxas info    : Used %s registers, used 1 barriers
ptxas info    : Compiling entry function '_ZN2fa10fwd_kernelILi128ELi8ELb0EEEv14CUtensorMap_stS1_S1_NS_9FwdParamsEi' for 'sm_103a'
ptxas info    : Function properties for _ZN2fa10fwd_kernelILi128ELi8ELb0EEEv14CUtensorMap_stS1_S1_NS_9FwdParamsEi
    72 bytes stack frame, 92 bytes spill stores, 160 bytes spill loads
ptxas info    : Used 168 registers, used 1 barriers
"""


def report(stack=0, st=0, ld=0, regs=168):
    return build.ptxas_report(REPORT % (stack, st, ld, regs))


def test_parse():
    r = report(8, 4, 36, 168)
    k = [n for n in r if "ILi128ELi0E" in n][0]
    assert r[k] == {"registers": 168, "spill_stores": 4, "spill_loads": 36}


def test_clean_report_passes():
    r = report()
    build.check_register_split(r)
    build.check_spills(r)  # the 8-of-32 polynomial split is exempt


def test_spill_in_default_forward_fails():
    with pytest.raises(RuntimeError, match="spills"):
        build.check_spills(report(8, 4, 36))


def test_wrong_register_count_fails():
    with pytest.raises(RuntimeError, match="registers per thread"):
        build.check_register_split(report(regs=160))


def test_backward_default_instance_has_a_spill_budget():
    text = REPORT.replace("fwd_kernelILi128ELi0ELb0E", "bwd_main_kernelILi128ELb0E") % (176, 172, 172, 128)
    build.check_spills(build.ptxas_report(text))  # within the budget
    with pytest.raises(RuntimeError, match="spills"):
        build.check_spills(build.ptxas_report(REPORT.replace("fwd_kernelILi128ELi0ELb0E", "bwd_main_kernelILi128ELb0E")
                                              % (400, 400, 400, 128)))
    with pytest.raises(RuntimeError, match="spills"):  # the deterministic instance has none
        build.check_spills(build.ptxas_report(REPORT.replace("fwd_kernelILi128ELi0ELb0E", "bwd_main_kernelILi128ELb1E")
                                              % (8, 4, 4, 128)))


def test_decoding_forward_needs_only_to_fit():
    dec = REPORT.replace("fwd_kernelILi128ELi0ELb0E", "fwd_kernelILi128ELi0ELb1E")
    r = build.ptxas_report(dec % (0, 0, 0, 148))
    build.check_register_split(r)  # no split in the decoding form: below the launch count is fine
    build.check_spills(r)
    with pytest.raises(RuntimeError, match="two CTAs per SM"):
        build.check_register_split(build.ptxas_report(dec % (0, 0, 0, 176)))
    build.check_spills(build.ptxas_report(dec % (96, 96, 140, 168)))  # within its budget
    with pytest.raises(RuntimeError, match="spills"):
        build.check_spills(build.ptxas_report(dec % (400, 400, 400, 168)))
