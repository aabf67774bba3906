"""Plain CPU oracle for the TQ1_0 mat-vec (test infrastructure only)."""
