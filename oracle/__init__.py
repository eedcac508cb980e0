"""CPU oracle for the deterministic attention backward: test infrastructure.

``attention``: fp64 softmax attention forward and backward from the textbook
definition.  ``dag_sim``: the DASH schedules written out from their
definitions, plus the DAG critical-path simulator that assigns chains to SMs.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  It shares no code with the CUDA library.
"""
