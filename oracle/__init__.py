"""Float64 CPU oracle of the MoE layer over one verification pass.

Test infrastructure only: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it; the product package never imports it.
"""
